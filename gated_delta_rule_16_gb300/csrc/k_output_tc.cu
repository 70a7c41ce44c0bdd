// k_output_tc.cu -- mapped two-chunk group output (SparseGDN Sec. 2.7,
// Eqs. 22-24) on tcgen05 tensor cores, for bf16 storage.
//
// One CTA per (group r, head pair p, sequence b): 128 query tokens (chunks
// c = 2r and c+1) against 128 key tokens.  TMEM holds three 128x128 fp32
// accumulators:
//   QK  = Q K^T                   (A: Q [tok][d] K-major; B: K [tok][d] K-major), shared by the pair
//   QS  = Q S_c                   (B: snapshot S^T [dv][d] bf16, K-major)
//   AU  = A U'                    (A: decayed, masked QK in bf16, K-major; B: U' [tok][dv] MN-major)
// per value head, where the mask/decay of A is
//   same chunk, j <= i : 2^(g_i - g_j);   i in c+1, j in c : 2^(g_i + gamma_c - g_j);   else 0
// and the epilogue forms O_i = (f 2^(g_i + shift_i) QS_i + AU_i) / sqrt(d) with
// f = 2^(P_c - P_(e+1)) the gap decay of the predecessor snapshot (Eq. 21) and
// shift_i = gamma_c for tokens of chunk c+1.  Operands arrive by TMA.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 512;  // 16 warps: 4 per TMEM lane quarter, 32 columns each
constexpr uint32_t kSlab = 16384;          // [128 rows][128 B]
constexpr uint32_t OFF_Q = 0;              // Q: 2 K-slabs
constexpr uint32_t OFF_K = 2 * kSlab;      // K: 2 K-slabs; later S^T of head 1 (2 K-slabs)
constexpr uint32_t OFF_S0 = 4 * kSlab;     // S^T of head 0: 2 K-slabs [128 dv][64 d]
constexpr uint32_t OFF_U0 = 6 * kSlab;     // U' of head 0: 2 MN-stacks [128 tok][64 dv]
constexpr uint32_t OFF_U1 = 8 * kSlab;     // U' of head 1
constexpr uint32_t OFF_A = 10 * kSlab;     // decayed masked A: 2 K-slabs [128 q][64 k]
constexpr uint32_t kOutSmem = 1024 + 12 * kSlab;
constexpr uint32_t TM_QK = 0, TM_QS = 128, TM_AU = 256, TM_QS1 = 384;  // QS of head 0 / head 1

struct OutParams {
    const float *g, *h0;
    const int4 *grp_info;   // per group: {snapshot slot, kind, decay head 0, decay head 1}
    __nv_bfloat16 *O;
    int32_t *status;
    int P_, T_, Nv, C, G;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__global__ void __launch_bounds__(kThreads, 1)
output_tc_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tK,
                 const __grid_constant__ CUtensorMap tU, const __grid_constant__ CUtensorMap tS,
                 const __grid_constant__ CUtensorMap tO, OutParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_qk_ld, bar_h_ld[2], bar_s[2], bar_qk_mma, bar_h_mma, bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    __shared__ float gs[2][128];
    __shared__ __align__(16) float colf[2][128];  // 2^(c_h - G_j): column factors of the group's decay mask
    __shared__ float cref[2], gmax_w[2][4], gmin_w[2][4];
    __shared__ int fact[2];          // 1: the mask factorises (the group's log-decay range is moderate)
    __shared__ float fscale[2];
    __shared__ int has_s[2], slot_s[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, seg = warp >> 2;  // TMEM lane quarter, 32-column segment
    const int row = quarter * 32 + lane;            // query token inside the group
    const int r = blockIdx.x, p = blockIdx.y, b = blockIdx.z;
    const int c0 = 2 * r;
    const bool two = c0 + 1 < a.C;
    const int t0 = c0 * kChunk;                     // first token of the group inside its sequence
    const int nvalid = min(2 * kChunk, a.T_ - t0);  // tokens of the group (a partial last chunk has fewer)
    const int64_t tok0 = (int64_t)b * a.T_ + t0;

    pdl_trigger();
    if (tid == 0) {  // the caller's Q and K go first: they do not depend on the kernels before
        mbar_init(&bar_qk_ld, 1);
        mbar_init(&bar_h_ld[0], 1);
        mbar_init(&bar_h_ld[1], 1);
        mbar_init(&bar_s[0], 1);
        mbar_init(&bar_s[1], 1);
        mbar_init(&bar_qk_mma, 1);
        mbar_init(&bar_h_mma, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        abort_s = 0;
        mbar_arrive_expect_tx(&bar_qk_ld, 4 * kSlab);
        tma_load_4d(sm + OFF_Q, &tQ, 0, p, t0, b, &bar_qk_ld);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_Q + kSlab, &tQ, 64, p, t0, b, &bar_qk_ld);
        tma_load_4d(sm + OFF_K, &tK, 0, p, t0, b, &bar_qk_ld);
        tma_load_4d(sm + OFF_K + kSlab, &tK, 64, p, t0, b, &bar_qk_ld);
    }
    for (int idx = tid; idx < 256; idx += kThreads) {  // tokens past the sequence's end: a finite g
        const int hh = idx >> 7, t = idx & 127;
        gs[hh][t] = a.g[(tok0 + min(t, nvalid - 1)) * a.Nv + 2 * p + hh];
    }
    if (warp == 0) tmem_alloc<512>(&tmem_base);
    pdl_wait();  // U', the entry-state table and the snapshots come from the kernels before
    if (tid == 0) {
        for (int hh = 0; hh < 2; ++hh) {
            uint8_t *ud = sm + (hh ? OFF_U1 : OFF_U0);
            mbar_arrive_expect_tx(&bar_h_ld[hh], 2 * kSlab);
            tma_load_4d(ud, &tU, 0, 2 * p + hh, t0, b, &bar_h_ld[hh]);
            tma_load_4d(ud + kSlab, &tU, 64, 2 * p + hh, t0, b, &bar_h_ld[hh]);
        }
    }
    if (tid < 2) {  // entry state of the group: one table load (kind 1 snapshot, 2 h0, 0 zero)
        const int4 info = a.grp_info[((int64_t)b * a.P_ + p) * a.G + r];
        const int hh = tid;
        has_s[hh] = info.y == 2 && !a.h0 ? 0 : info.y;
        slot_s[hh] = info.x;
        fscale[hh] = __int_as_float(hh ? info.w : info.z);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;

    // Decay mask of the group.  With G_t the log2 decay accumulated from the group's start
    // (chunk c: g_t; chunk c+1: gamma_c + g_t), every kept entry (j <= i, same chunk or the
    // cross block) is 2^(G_i - G_j).  When the group's range of G is moderate the mask is a
    // product of a row factor 2^(G_i - c) and a column factor 2^(c - G_j), c the middle of the
    // range, so the A tile needs no per-element exp2; otherwise it falls back to one exp2 each.
    auto gcum = [&](int hh, int t) { return t < 64 ? gs[hh][t] : gs[hh][63] + gs[hh][t]; };
    if (tid < 256) {
        const int hh = tid >> 7, t = tid & 127, wi = (tid >> 5) & 3;
        const bool used = t < (two ? 128 : 64);
        float mx = used ? gcum(hh, t) : -INFINITY, mn = used ? gcum(hh, t) : INFINITY;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (lane == 0) { gmax_w[hh][wi] = mx; gmin_w[hh][wi] = mn; }
    }
    __syncthreads();
    if (tid < 256) {
        const int hh = tid >> 7, t = tid & 127;
        const float mx = fmaxf(fmaxf(gmax_w[hh][0], gmax_w[hh][1]), fmaxf(gmax_w[hh][2], gmax_w[hh][3]));
        const float mn = fminf(fminf(gmin_w[hh][0], gmin_w[hh][1]), fminf(gmin_w[hh][2], gmin_w[hh][3]));
        const float c = 0.5f * (mx + mn);
        colf[hh][t] = ex2(c - gcum(hh, t));
        if (t == 0) {
            cref[hh] = c;
            fact[hh] = (mx - mn) <= 200.f;  // both factors stay within 2^(+-100)
        }
    }

    // initial-state path (no predecessor event, h0 given): S^T = h0^T in bf16, K-major slabs
    auto fill_h0 = [&](int hh, uint8_t *dst) {
        const float *src = a.h0 + ((int64_t)b * a.Nv + 2 * p + hh) * (kDim * kDim);
        for (int idx = tid; idx < kDim * 16; idx += kThreads) {  // (dv row, 8-wide d chunk)
            const int dv = idx & 127, ch = idx >> 7;
            float v[8];
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2) v[q2] = src[(ch * 8 + q2) * kDim + dv];
            st_sw128_8(dst + (ch >> 3) * kSlab, dv, (ch & 7) * 8, v);
        }
        fence_async_smem();
    };

    if (tid == 0 && has_s[0] == 1) {
        mbar_arrive_expect_tx(&bar_s[0], 2 * kSlab);
        tma_load_3d(sm + OFF_S0, &tS, 0, slot_s[0] * 2 * kDim, 0, &bar_s[0]);
        tma_load_3d(sm + OFF_S0 + kSlab, &tS, 64, slot_s[0] * 2 * kDim, 0, &bar_s[0]);
    }
    if (has_s[0] == 2) fill_h0(0, sm + OFF_S0);
    __syncthreads();

    const uint32_t id_kk = idesc_bf16(128, 128, false, false);
    const uint32_t id_km = idesc_bf16(128, 128, false, true);
    const float inv_sqrt_d = rsqrtf((float)kDim);
    bool ok = true;
    bool s1_issued = false;  // thread 0
    if (tid == 0) {
        ok = mbar_wait(&bar_qk_ld, 0);
        if (ok) {
            tc_fence_after();
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tbase + TM_QK, kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                         kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id_kk, ks > 0);
            mma_commit(&bar_qk_mma);
        }
        if (!ok) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
    }
    __syncthreads();

    for (int hh = 0; hh < 2 && !abort_s; ++hh) {
        // 1. A_h from QK (waits for the QK MMA; for head 1 also for head 0's AU MMA to free the A tile)
        if (!mbar_wait(hh == 0 ? &bar_qk_mma : &bar_h_mma, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
        tc_fence_after();
        if (tid == 0 && !abort_s) {
            if (hh == 0 && has_s[1] == 1) {  // the K tile is free once QK is done: head 1's snapshot goes there
                mbar_arrive_expect_tx(&bar_s[1], 2 * kSlab);
                tma_load_3d(sm + OFF_K, &tS, 0, (slot_s[1] * 2 + 1) * kDim, 0, &bar_s[1]);
                tma_load_3d(sm + OFF_K + kSlab, &tS, 64, (slot_s[1] * 2 + 1) * kDim, 0, &bar_s[1]);
                s1_issued = true;
            }
            // QS of this head needs only Q and its entry state (head 1 from h0: written with its A
            // tile, so issued with AU below): issue it now, while the A tile is built
            const bool qs_now = has_s[hh] == 1 || (hh == 0 && has_s[0] == 2);
            if (qs_now) {
                if (has_s[hh] == 1 && !mbar_wait(&bar_s[hh], 0)) {
                    abort_s = 1;
                    atomicOr(a.status, kStatusTimeout);
                } else {
                    uint8_t *st = sm + (hh ? OFF_K : OFF_S0);
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tbase + (hh ? TM_QS1 : TM_QS), kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                                 kmajor_desc(smem_addr(st), ks, kSlab), id_kk, ks > 0);
                }
            }
        }
        {
            const int ci = row >> 6;
            const float Gi = gcum(hh, row);
            const bool zero_row = ci == 1 && !two;  // a final single-chunk group has no second chunk
            float qk[32];
            const int j0 = 32 * seg;
            tmem_ld32(tmem_addr(tbase, quarter * 32, TM_QK + j0), qk);
            tmem_ld_wait();
            float w[32];
            if (fact[hh]) {
                const float ef = ex2(Gi - cref[hh]);
                const float4 *cf = reinterpret_cast<const float4 *>(colf[hh] + j0);
#pragma unroll
                for (int t4 = 0; t4 < 8; ++t4) {
                    const float4 f = cf[t4];
                    const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = 4 * t4 + u;
                        w[t] = (j0 + t <= row && !zero_row) ? qk[t] * ef * fv[u] : 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    w[t] = (j0 + t <= row && !zero_row) ? qk[t] * ex2(Gi - gcum(hh, j0 + t)) : 0.f;
            }
#pragma unroll
            for (int t0 = 0; t0 < 32; t0 += 8)
                st_sw128_8(sm + OFF_A + (seg >> 1) * kSlab, row, 32 * (seg & 1) + t0, &w[t0]);
        }
        if (hh == 1 && has_s[1] == 2) fill_h0(1, sm + OFF_K);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;
        // 2. QS_h and AU_h
        if (tid == 0) {
            const bool landed = mbar_wait(&bar_h_ld[hh], 0) && !(has_s[hh] == 1 && !mbar_wait(&bar_s[hh], 0));
            if (!landed) {
                abort_s = 1;
                atomicOr(a.status, kStatusTimeout);
            } else {
                tc_fence_after();
                uint8_t *ut = sm + (hh ? OFF_U1 : OFF_U0);
                if (hh == 1 && has_s[1] == 2)  // head 1 from h0: its state was written with the A tile
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tbase + TM_QS1, kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                                 kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id_kk, ks > 0);
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_AU, kmajor_desc(smem_addr(sm + OFF_A), ks, kSlab),
                             mnmajor_desc(smem_addr(ut), ks, kSlab), id_km, ks > 0);
                mma_commit(&bar_h_mma);
            }
        }
        __syncthreads();
        if (abort_s) break;
        if (!mbar_wait(&bar_h_mma, hh)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
        tc_fence_after();
        // 3. epilogue of head hh: O rows staged (bf16, 128B-swizzled) in the U' tile
        //    this head no longer needs, then written by one TMA store
        {
            const float f = fscale[hh] * ex2(gs[hh][row] + (row >= 64 ? gs[hh][63] : 0.f));
            const bool has = has_s[hh] != 0;
            uint8_t *stage = sm + (hh ? OFF_U1 : OFF_U0) + (seg >> 1) * kSlab;
            {
                float qs[32], au[32];
                const int col = 32 * seg;
                tmem_ld32(tmem_addr(tbase, quarter * 32, TM_AU + col), au);
                if (has) tmem_ld32(tmem_addr(tbase, quarter * 32, (hh ? TM_QS1 : TM_QS) + col), qs);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t) au[t] = ((has ? f * qs[t] : 0.f) + au[t]) * inv_sqrt_d;
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(stage, row, 32 * (seg & 1) + 8 * v8, &au[8 * v8]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            uint8_t *stage = sm + (hh ? OFF_U1 : OFF_U0);
            tma_store_4d(&tO, 0, 2 * p + hh, t0, b, stage);  // rows past the sequence's end are clipped
            tma_store_4d(&tO, 64, 2 * p + hh, t0, b, stage + kSlab);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_read();  // the stores only need their shared-memory sources before exit
    if (abort_s && tid == 0) {
        // let every copy and MMA issued so far land before the CTA releases its memory
        mbar_wait(&bar_qk_ld, 0);
        mbar_wait(&bar_h_ld[0], 0);
        mbar_wait(&bar_h_ld[1], 0);
        if (has_s[0] == 1) mbar_wait(&bar_s[0], 0);
        if (s1_issued) mbar_wait(&bar_s[1], 0);
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tbase);
}

}  // namespace

cudaError_t launch_output_tc(const Problem &pb, const Workspace &ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tQ, tK, tU, tS, tO;
    const uint64_t snap_rows = (uint64_t)(ws.snap_cap > 0 ? ws.snap_cap : 1) * 2 * kDim;
    if (!make_tmap_tokens(&tQ, pb.q, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tU, ws.U, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_bf16_3d(&tS, ws.snap, kDim, snap_rows, 1, kDim * 2, snap_rows * kDim * 2, 64, 128, 1) ||
        !make_tmap_tokens(&tO, pb.o, pb.Nv, pb.T, pb.B, 64, 128))
        return cudaErrorInvalidValue;
    OutParams a;
    a.g = pb.g; a.h0 = pb.h0; a.grp_info = (const int4 *)ws.grp_info;
    a.O = (__nv_bfloat16 *)pb.o; a.status = ws.counts + 2;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.G = pb.G;
    cudaFuncSetAttribute(output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem);
    return launch_kernel(pb.pdl, output_tc_kernel, dim3(pb.G, pb.P, pb.B), kThreads, kOutSmem, pb.stream, tQ, tK, tU,
                         tS, tO, a);
}

}  // namespace gdn
