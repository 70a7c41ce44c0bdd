// k_output_tc.cu -- mapped two-chunk group output (SparseGDN Sec. 2.7,
// Eqs. 22-24) on tcgen05 tensor cores, for bf16 storage.
//
// One CTA per (group r, value head h, sequence b): 128 query tokens (chunks
// c = 2r and c+1) against 128 key tokens; 256 threads, ~68 KB of shared memory, 128
// TMEM columns and at most 80 registers a thread, so three CTAs share an SM and keep
// enough loads in flight for the kernel's bytes (the two heads of a pair are adjacent
// CTAs; the second read of their Q and K tiles comes from L2).
//   QK  = Q K^T                   (A: Q [tok][d] K-major; B: K [tok][d] K-major)
//   O   = (f Q) S_c + A U'        (one accumulator: B of the first product the snapshot
//                                  S^T [dv][d] bf16, K-major; of the second U' [tok][dv] MN-major)
// where the mask/decay of A is
//   same chunk, j <= i : 2^(g_i - g_j);   i in c+1, j in c : 2^(g_i + gamma_c - g_j);   else 0
// and row i of Q is scaled, in bf16, by f_i = 2^(P_c - P_(e+1)) 2^(g_i + shift_i): the gap decay
// of the predecessor snapshot (Eq. 21) times the decay into token i (shift_i = gamma_c for tokens
// of chunk c+1).  O leaves scaled by 1/sqrt(d).  Operands arrive by TMA.
// Shared memory over the CTA's life (two 32 KB tiles):
//   [0, 32K)    Q (QK) -> f Q (QS) -> the A tile
//   [32K, 64K)  K (QK) -> the entry state S^T -> U' -> O staging
// The A values wait in registers (packed bf16) from QK until QS has read the scaled Q; the
// entry state and U' each load once the product before has read that tile.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 256;  // 8 warps: 2 per TMEM lane quarter, 64 columns each
constexpr uint32_t kSlab = 16384;          // [128 rows][128 B]
constexpr uint32_t OFF_Q = 0;              // Q, rows scaled by the state factor for QS; then the A tile
constexpr uint32_t OFF_K = 2 * kSlab;      // K; then the entry state S^T; then U' [128 tok][64 dv] x 2; then O
constexpr uint32_t kOutSmem = 1024 + 4 * kSlab;
constexpr uint32_t TM_O = 0;  // QK, then the output accumulator f Q S + A U' (128 columns)

struct OutParams {
    const float *g, *h0;
    const int4 *grp_info;   // per group: {snapshot slot, kind, decay head 0, decay head 1}
    __nv_bfloat16 *O;
    int32_t *status;
    const int32_t *row_pair;  // non-NULL: blockIdx.y is CSR row row0 + y (pair row_pair[row0 + y])
    int row0;
    int expanded;             // entry states by group (slot (b P + p) G + r), not through the map
    int P_, T_, Nv, C, G;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads, 3)
output_tc_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tK,
                 const __grid_constant__ CUtensorMap tU, const __grid_constant__ CUtensorMap tS,
                 const __grid_constant__ CUtensorMap tO, OutParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_qk_ld, bar_u_ld, bar_s, bar_qk, bar_qs, bar_au, bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    __shared__ float gs[128];
    __shared__ __align__(16) float colf[128];  // 2^(c - G_j): column factors of the group's decay mask
    __shared__ float cref, gmax_w[4], gmin_w[4];
    __shared__ int fact;  // 1: the mask factorises (the group's log-decay range is moderate)
    __shared__ float fscale;
    __shared__ int has_s, s_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter; which 64 of 128 columns
    const int row = quarter * 32 + lane;             // query token inside the group
    const int hh = blockIdx.x & 1, r = blockIdx.x >> 1;
    // (row_pair is complete before this kernel's stream forked from the compaction's)
    const int pr = a.row_pair ? a.row_pair[a.row0 + blockIdx.y] : 0;
    const int p = a.row_pair ? pr % a.P_ : (int)blockIdx.y, b = a.row_pair ? pr / a.P_ : (int)blockIdx.z;
    const int h = 2 * p + hh;
    const int c0 = 2 * r;
    const bool two = c0 + 1 < a.C;
    const int t0 = c0 * kChunk;                     // first token of the group inside its sequence
    const int nvalid = min(2 * kChunk, a.T_ - t0);  // tokens of the group (a partial last chunk has fewer)
    const int64_t tok0 = (int64_t)b * a.T_ + t0;

    pdl_trigger();
    if (tid == 0) {  // the caller's Q and K go first: they do not depend on the kernels before
        mbar_init(&bar_qk_ld, 1);
        mbar_init(&bar_u_ld, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_qk, 1);
        mbar_init(&bar_qs, 1);
        mbar_init(&bar_au, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        abort_s = 0;
        mbar_arrive_expect_tx(&bar_qk_ld, 4 * kSlab);
        tma_load_4d(sm + OFF_Q, &tQ, 0, p, t0, b, &bar_qk_ld);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_Q + kSlab, &tQ, 64, p, t0, b, &bar_qk_ld);
        tma_load_4d(sm + OFF_K, &tK, 0, p, t0, b, &bar_qk_ld);
        tma_load_4d(sm + OFF_K + kSlab, &tK, 64, p, t0, b, &bar_qk_ld);
    }
    if (tid < 128) gs[tid] = a.g[(tok0 + min(tid, nvalid - 1)) * a.Nv + h];  // past the end: a finite g
    if (warp == 0) tmem_alloc<128>(&tmem_base);
    pdl_wait();  // U', the entry-state table and the snapshots come from the kernels before
    if (tid == 0) {  // entry state of the group: one table load (kind 1 snapshot, 2 h0, 0 zero)
        const int4 info = a.grp_info[((int64_t)b * a.P_ + p) * a.G + r];
        const int kind = info.y == 2 && !a.h0 ? 0 : info.y;
        has_s = kind;
        fscale = __int_as_float(hh ? info.w : info.z);
        s_slot = a.expanded ? (b * a.P_ + p) * a.G + r : info.x;
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
    auto gcum = [&](int t) { return t < 64 ? gs[t] : gs[63] + gs[t]; };
    if (tid < 128) {
        const bool used = tid < (two ? 128 : 64);
        float mx = used ? gcum(tid) : -INFINITY, mn = used ? gcum(tid) : INFINITY;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (lane == 0) { gmax_w[warp] = mx; gmin_w[warp] = mn; }
    }
    __syncthreads();
    if (tid < 128) {
        const float mx = fmaxf(fmaxf(gmax_w[0], gmax_w[1]), fmaxf(gmax_w[2], gmax_w[3]));
        const float mn = fminf(fminf(gmin_w[0], gmin_w[1]), fminf(gmin_w[2], gmin_w[3]));
        const float c = 0.5f * (mx + mn);
        colf[tid] = ex2(c - gcum(tid));
        if (tid == 0) {
            cref = c;
            fact = (mx - mn) <= 200.f;  // both factors stay within 2^(+-100)
        }
    }

    const uint32_t id_kk = idesc_bf16(128, 128, false, false);
    const uint32_t id_km = idesc_bf16(128, 128, false, true);
    const float inv_sqrt_d = rsqrtf((float)kDim);
    const int kind = has_s;
    bool s_issued = false, s_wait_ok = true, u_issued = false;  // thread 0
    if (tid == 0) {  // QK
        if (!mbar_wait(&bar_qk_ld, 0)) {
            abort_s = 1;
            atomicOr(a.status, kStatusTimeout);
        } else {
            tc_fence_after();
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tbase + TM_O, kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                         kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id_kk, ks > 0);
            mma_commit(&bar_qk);
        }
    }
    __syncthreads();  // publishes abort_s and the mask factors
    // 1. A from QK, in registers as packed bf16: thread (row, half) covers key columns 64 half ..
    uint32_t apk[32];
    if (!abort_s && !mbar_wait(&bar_qk, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
    tc_fence_after();
    {
        const float Gi = gcum(row);
        const bool zero_row = row >= 64 && !two;  // a final single-chunk group has no second chunk
        const float ef = ex2(Gi - cref);
        const bool fct = fact != 0;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
            const int j0 = 64 * half + 16 * s4;
            float qk[16];
            tmem_ld16(tmem_addr(tbase, quarter * 32, TM_O + j0), qk);
            tmem_ld_wait();
            float w[16];
            if (fct) {
                const float4 *cf = reinterpret_cast<const float4 *>(colf + j0);
#pragma unroll
                for (int t4 = 0; t4 < 4; ++t4) {
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
                for (int t = 0; t < 16; ++t)
                    w[t] = (j0 + t <= row && !zero_row) ? qk[t] * ex2(Gi - gcum(j0 + t)) : 0.f;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) apk[8 * s4 + t] = pack_bf16(w[2 * t], w[2 * t + 1]);
        }
    }
    tc_fence_before();
    __syncthreads();  // QK has read K and every thread has read QK
    // 2. the entry state takes K's place; the rows of Q are scaled by the state's factor
    //    f_i = 2^(P_c - P_(e+1)) 2^(g_i + shift_i), so that one accumulator holds f Q S + A U'
    if (tid == 0 && !abort_s && kind == 1) {
        mbar_arrive_expect_tx(&bar_s, 2 * kSlab);
        tma_load_3d(sm + OFF_K, &tS, 0, (s_slot * 2 + hh) * kDim, 0, &bar_s);
        tma_load_3d(sm + OFF_K + kSlab, &tS, 64, (s_slot * 2 + hh) * kDim, 0, &bar_s);
        s_issued = true;
    }
    if (kind == 2) {  // initial-state path (no predecessor event, h0 given): S^T = h0^T in bf16, K-major slabs
        const float *src = a.h0 + ((int64_t)b * a.Nv + h) * (kDim * kDim);
        for (int idx = tid; idx < kDim * 16; idx += kThreads) {  // (dv row, 8-wide d chunk)
            const int dv = idx & 127, ch = idx >> 7;
            float v[8];
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2) v[q2] = src[(ch * 8 + q2) * kDim + dv];
            st_sw128_8(sm + OFF_K + (ch >> 3) * kSlab, dv, (ch & 7) * 8, v);
        }
    }
    if (kind != 0) {  // thread (row, half): the row's 64 columns of Q in slab `half`
        const float f = fscale * ex2(gs[row] + (row >= 64 ? gs[63] : 0.f));
        uint8_t *slab = sm + OFF_Q + half * kSlab;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            uint4 *ptr = reinterpret_cast<uint4 *>(slab + sw128_offset(row, 8 * c8));
            const uint4 q = *ptr;
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&qw[e]);
                o4[e] = pack_bf16(__low2float(v) * f, __high2float(v) * f);
            }
            *ptr = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // 3. QS = (f Q) S starts the accumulator (no entry state: nothing to add)
    if (tid == 0 && !abort_s) {
        if (kind != 0) {
            if (kind == 1 && !mbar_wait(&bar_s, 0)) {
                s_wait_ok = false;
                abort_s = 1;
                atomicOr(a.status, kStatusTimeout);
            } else {
                tc_fence_after();
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_O, kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                             kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id_kk, ks > 0);
            }
        }
        mma_commit(&bar_qs);  // also without QS: arrives at once (QK is done)
    }
    // 4. QS has read the scaled Q and the state: U' takes K's place, the A tile Q's
    if (!abort_s && !mbar_wait(&bar_qs, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
    if (tid == 0 && !abort_s) {
        mbar_arrive_expect_tx(&bar_u_ld, 2 * kSlab);
        tma_load_4d(sm + OFF_K, &tU, 0, t0, h, b, &bar_u_ld);
        tma_load_4d(sm + OFF_K + kSlab, &tU, 64, t0, h, b, &bar_u_ld);
        u_issued = true;
    }
    {
        uint8_t *slab = sm + OFF_Q + half * kSlab;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
            *reinterpret_cast<uint4 *>(slab + sw128_offset(row, 8 * c8)) =
                make_uint4(apk[4 * c8], apk[4 * c8 + 1], apk[4 * c8 + 2], apk[4 * c8 + 3]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // 5. AU = A U' added onto QS
    if (tid == 0 && !abort_s) {
        if (!mbar_wait(&bar_u_ld, 0)) {
            abort_s = 1;
            atomicOr(a.status, kStatusTimeout);
        } else {
            tc_fence_after();
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tbase + TM_O, kmajor_desc(smem_addr(sm + OFF_Q), ks, kSlab),
                         mnmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id_km, kind != 0 || ks > 0);
            mma_commit(&bar_au);
        }
    }
    __syncthreads();
    if (!abort_s && !mbar_wait(&bar_au, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
    tc_fence_after();
    // 6. epilogue: O rows staged (bf16, 128B-swizzled) over U' (read by now), one TMA store
    {
        uint8_t *stage = sm + OFF_K + half * kSlab;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            float o[32];
            tmem_ld32(tmem_addr(tbase, quarter * 32, TM_O + 64 * half + 32 * s2), o);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] *= inv_sqrt_d;
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(stage, row, 32 * s2 + 8 * v8, &o[8 * v8]);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && !abort_s) {
        tma_store_4d(&tO, 0, h, t0, b, sm + OFF_K);  // rows past the sequence's end are clipped
        tma_store_4d(&tO, 64, h, t0, b, sm + OFF_K + kSlab);
        bulk_commit();
    }
    if (tid == 0) bulk_wait_read();  // the stores only need their shared-memory sources before exit
    if (abort_s && tid == 0) {
        // let every copy and MMA issued so far land before the CTA releases its memory
        mbar_wait(&bar_qk_ld, 0);
        if (s_issued && s_wait_ok) mbar_wait(&bar_s, 0);
        if (u_issued) mbar_wait(&bar_u_ld, 0);
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<128>(tbase);
}

}  // namespace

cudaError_t launch_output_tc(const Problem &pb, const Workspace &ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tQ, tK, tU, tS, tO;
    const uint64_t snap_rows = (uint64_t)(ws.snap_cap > 0 ? ws.snap_cap : 1) * 2 * kDim;
    if (!make_tmap_tokens(&tQ, pb.q, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_headmajor(&tU, ws.U, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_bf16_3d(&tS, ws.snap, kDim, snap_rows, 1, kDim * 2, snap_rows * kDim * 2, 64, 128, 1) ||
        !make_tmap_tokens(&tO, pb.o, pb.Nv, pb.T, pb.B, 64, 128))
        return cudaErrorInvalidValue;
    OutParams a;
    a.g = pb.g; a.h0 = pb.h0; a.grp_info = (const int4 *)ws.grp_info;
    a.O = (__nv_bfloat16 *)pb.o; a.status = ws.counts + 2;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.G = pb.G;
    a.row_pair = pb.nrows > 0 ? pb.row_pair : nullptr;
    a.row0 = pb.row0;
    a.expanded = pb.states_expanded;
    cudaFuncSetAttribute(output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem);
    const dim3 grid = pb.nrows > 0 ? dim3(2 * pb.G, pb.nrows, 1) : dim3(2 * pb.G, pb.P, pb.B);
    return launch_kernel(pb.pdl, output_tc_kernel, grid, kThreads, kOutSmem, pb.stream, tQ, tK, tU, tS, tO, a);
}

}  // namespace gdn
