// k_intra_tc.cu -- intra-chunk step (SparseGDN Sec. 2.3, Eqs. 5-9) on tcgen05
// tensor cores, for bf16 storage.
//
// One CTA per (group of two chunks, head pair, sequence): 128 tokens.
//   Gram  G = K K^T [128 x 128]        (A = B = the K tile, K-major, by TMA), shared by the pair
// per value head:
//   A_Delta[t,s] = beta_t G[t,s] 2^(g_t - g_s), s < t in the same chunk; M = I + A_Delta
//   C = M^-1 (exact) or the block-adjacent approximation (Eq. 7), fp32 on CUDA cores:
//       C_ii = M_ii^-1 (forward substitution), C_ij = -C_ii sum_{k=j}^{i-1} M_ik C_kj
//   U = C diag(beta) V                  (A: C diag(beta) bf16, block-diagonal over the
//                                        two chunks, K-major; B: V [tok][dv] MN-major by TMA)
//   s = ||U[48:64,:]||_F (Tail-16 write score)
//   W = C diag(beta 2^g) K for the chunks that are events (Eq. 15): A = C-bar bf16,
//       block-diagonal, K-major; B = the K tile read as MN-major (token rows, d
//       columns: the same bytes as the K-major Gram operand).  W is written at the
//       event's index, so it is never built for skipped chunks.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 512;  // 16 warps: 4 per TMEM lane quarter, 32 columns each
constexpr uint32_t kSlab = 16384;
constexpr uint32_t OFF_K = 0;            // K tile: 2 K-slabs [128 tok][64 d]
constexpr uint32_t OFF_V = 2 * kSlab;    // V tiles of the two heads: 2 MN-stacks [128 tok][64 dv] each
constexpr uint32_t OFF_A = 6 * kSlab;    // C diag(beta) bf16: 2 K-slabs [128 t][64 s]
constexpr uint32_t OFF_F = 8 * kSlab;    // fp32 work area
// Row stride of the fp32 64x64 tiles: 68 floats keeps rows 16-byte aligned, and a
// 16-byte access by eight threads owning eight consecutive rows (one shared-memory
// wavefront) touches 8 x 4 distinct banks.
constexpr int MS = kChunk + 4;
constexpr uint32_t F_M = 0;                              // [2][64][68] M
constexpr uint32_t F_C = F_M + 2 * kChunk * MS * 4;      // [2][64][68] C
constexpr uint32_t F_T = F_C + 2 * kChunk * MS * 4;      // [2][3][256] block products
constexpr uint32_t F_B = F_T + 2 * 3 * 256 * 4;          // [2 heads][128] beta
constexpr uint32_t F_G = F_B + 2 * 128 * 4;              // [2 heads][128] g
constexpr uint32_t F_BG = F_G + 2 * 128 * 4;             // [128] beta 2^g of the current head
constexpr uint32_t F_S = F_BG + 128 * 4;                 // [2] score partial sums
constexpr uint32_t kIntraTcSmem = 1024 + OFF_F + F_S + 64;
constexpr uint32_t TM_G = 0, TM_U = 128, TM_W = 256;

struct IntraParams {
    const float *beta, *g;
    const int32_t *ev_of;   // NULL: no W here (online selection builds W later from C-bar)
    __nv_bfloat16 *U, *W;
    __nv_bfloat16 *cbar;    // non-NULL: write the compact C-bar blocks [B,Nv,C,nblk,16,16] (bf16)
    float *score;
    int32_t *status;
    int P_, T_, Nv, C, nblk, exact, tail;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 &b) {
    acc.x += a * b.x;
    acc.y += a * b.y;
    acc.z += a * b.z;
    acc.w += a * b.w;
}

// Off-diagonal 16x16 blocks at distance OFF of both chunks' C (Eq. 7 generalised):
// C_ij = -C_ii (sum_{k=j}^{i-1} M_ik C_kj), i = j + OFF, once every block closer to
// the diagonal is known.  Thread (chunk, block, row, column quad): 4 outputs from
// 16-byte shared-memory loads (a row of M or C_ii, a quad of a row of C or T).
template <int OFF>
__device__ __forceinline__ void offdiag_blocks(const float *Ms, float *Cs, float *Tb, int tid) {
    constexpr int NB = 4 - OFF;
    const bool act = tid < 2 * NB * 64;
    const int cc = tid / (NB * 64), rem = tid % (NB * 64);
    const int bi = rem >> 6, rr = (rem >> 2) & 15, q4 = (rem & 3) * 4;
    const int ib = bi + OFF, jb = bi;
    if (act) {  // T = sum_k M_{ib,k} C_{k,jb}: row rr, columns q4 .. q4+3
        const float *Mr = Ms + (cc * kChunk + ib * kBlk + rr) * MS + jb * kBlk;
        const float *Cc = Cs + (cc * kChunk + jb * kBlk) * MS + jb * kBlk + q4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k4 = 0; k4 < kBlk * OFF; k4 += 4) {
            const float4 m = ld4(Mr + k4);
            fma4(acc, m.x, ld4(Cc + (k4 + 0) * MS));
            fma4(acc, m.y, ld4(Cc + (k4 + 1) * MS));
            fma4(acc, m.z, ld4(Cc + (k4 + 2) * MS));
            fma4(acc, m.w, ld4(Cc + (k4 + 3) * MS));
        }
        *reinterpret_cast<float4 *>(Tb + (cc * NB + bi) * 256 + rr * 16 + q4) = acc;
    }
    __syncthreads();
    if (act) {  // C_{ib,jb} = -C_{ib,ib} T
        float *Cr = Cs + (cc * kChunk + ib * kBlk + rr) * MS;
        const float *Tt = Tb + (cc * NB + bi) * 256 + q4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m4 = 0; m4 < kBlk; m4 += 4) {
            const float4 c = ld4(Cr + ib * kBlk + m4);
            fma4(acc, c.x, ld4(Tt + (m4 + 0) * 16));
            fma4(acc, c.y, ld4(Tt + (m4 + 1) * 16));
            fma4(acc, c.z, ld4(Tt + (m4 + 2) * 16));
            fma4(acc, c.w, ld4(Tt + (m4 + 3) * 16));
        }
        *reinterpret_cast<float4 *>(Cr + jb * kBlk + q4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
intra_tc_kernel(const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
                const __grid_constant__ CUtensorMap tU, const __grid_constant__ CUtensorMap tW, IntraParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_ld, bar_g, bar_u, bar_w, bar_drain;
    __shared__ int ev_s[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    float *Ms = reinterpret_cast<float *>(sm + OFF_F + F_M);
    float *Cs = reinterpret_cast<float *>(sm + OFF_F + F_C);
    float *Tb = reinterpret_cast<float *>(sm + OFF_F + F_T);
    float *bet2 = reinterpret_cast<float *>(sm + OFF_F + F_B);
    float *gg2 = reinterpret_cast<float *>(sm + OFF_F + F_G);
    float *bgs = reinterpret_cast<float *>(sm + OFF_F + F_BG);
    float *ssum = reinterpret_cast<float *>(sm + OFF_F + F_S);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, seg = warp >> 2;  // TMEM lane quarter, 32-column segment
    const int row = quarter * 32 + lane;            // token inside the group
    const int ct = row >> 6, tl = row & 63;
    const int r = blockIdx.x, p = blockIdx.y, b = blockIdx.z;
    const int c0 = 2 * r;
    const int nch = c0 + 1 < a.C ? 2 : 1;
    const int t0 = c0 * kChunk;                        // first token of the group inside its sequence
    const int nvalid = min(2 * kChunk, a.T_ - t0);     // tokens of the group (a partial last chunk has fewer)
    const int64_t tok0 = (int64_t)b * a.T_ + t0;
    // Tail-W window of this thread's row: the last W valid rows of its chunk (rows past the
    // sequence's end need no exclusion: beta = 0 there makes their U rows exactly zero)
    const int nrow = min(kChunk, nvalid - kChunk * ct);
    const bool in_tail = tl >= nrow - a.tail;

    pdl_trigger();
    if (tid == 0) {  // barriers, then the tiles: the loads overlap the set-up below
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_u, 1);
        mbar_init(&bar_w, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        abort_s = 0;
        mbar_arrive_expect_tx(&bar_ld, 6 * kSlab);
        tma_load_4d(sm + OFF_K, &tK, 0, p, t0, b, &bar_ld);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_K + kSlab, &tK, 64, p, t0, b, &bar_ld);
        for (int hh = 0; hh < 2; ++hh) {
            uint8_t *vd = sm + OFF_V + hh * 2 * kSlab;
            tma_load_4d(vd, &tV, 0, 2 * p + hh, t0, b, &bar_ld);
            tma_load_4d(vd + kSlab, &tV, 64, 2 * p + hh, t0, b, &bar_ld);
        }
    }
    if (tid < 256) {  // beta and g of both heads, fetched once while the tiles load
        // tokens past the sequence's end: beta = 0 (no write, no correction) and a finite g
        const int hh = tid >> 7, t = tid & 127;
        const bool valid = t < nvalid;
        const int64_t gi = (tok0 + min(t, nvalid - 1)) * a.Nv + 2 * p + hh;
        bet2[tid] = valid ? a.beta[gi] : 0.f;
        gg2[tid] = a.g[gi];
    }
    if (warp == 0) tmem_alloc<512>(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    if (tid == 0) {
        if (!mbar_wait(&bar_ld, 0)) {
            abort_s = 1;
            atomicOr(a.status, kStatusTimeout);
        } else {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, false, false);
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tbase + TM_G, kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab),
                         kmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id, ks > 0);
            mma_commit(&bar_g);
        }
    }
    __syncthreads();
    const int max_off = a.exact ? 3 : 1;
    for (int hh = 0; hh < 2 && !abort_s; ++hh) {
        const int h = 2 * p + hh;
        const float *bet = bet2 + 128 * hh;
        const float *gg = gg2 + 128 * hh;
        if (tid < 128) bgs[tid] = bet[tid] * ex2(gg[tid]);
        if (tid < 2) ssum[tid] = 0.f;
        __syncthreads();
        // 1. M from the Gram block of the row's chunk: thread (row, half) covers 32 columns
        if (hh == 0 && !mbar_wait(&bar_g, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
        tc_fence_after();
        if (seg < 2) {
            const int hf = seg;
            float gv[32];
            tmem_ld32(tmem_addr(tbase, quarter * 32, TM_G + 64 * ct + 32 * hf), gv);
            tmem_ld_wait();
            const float bt = bet[row], gt = gg[row];
            float4 *mrow = reinterpret_cast<float4 *>(Ms + (ct * kChunk + tl) * MS + 32 * hf);
#pragma unroll
            for (int q2 = 0; q2 < 32; ++q2) {
                const int s = 32 * hf + q2;
                gv[q2] = s < tl ? bt * gv[q2] * ex2(gt - gg[64 * ct + s]) : (s == tl ? 1.f : 0.f);
            }
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                mrow[q4] = make_float4(gv[4 * q4], gv[4 * q4 + 1], gv[4 * q4 + 2], gv[4 * q4 + 3]);
        }
        __syncthreads();
        // 2. solve.  Diagonal 16x16 blocks by forward substitution: warp w < 4 takes
        //    blocks 2w and 2w+1 (8 blocks: 2 chunks x 4), one lane per column, the
        //    column of C_ii in registers and the rows of M_ii broadcast from shared memory:
        //    C_ii[i][j] = -sum_{s<i} M_ii[i][s] C_ii[s][j]   (C_ii[s][j] = 0 for s < j, 1 for s = j)
        if (warp < 4) {
            const int blk = 2 * warp + (lane >> 4), j = lane & 15;
            const int cc = blk >> 2, r0 = (blk & 3) * kBlk;
            const float *Mb = Ms + (cc * kChunk + r0) * MS + r0;
            float x[kBlk];
#pragma unroll
            for (int i2 = 0; i2 < kBlk; ++i2) x[i2] = i2 == j ? 1.f : 0.f;
#pragma unroll
            for (int i2 = 1; i2 < kBlk; ++i2) {
                float acc = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < i2; ++s2) acc += Mb[i2 * MS + s2] * x[s2];
                if (i2 > j) x[i2] = -acc;
            }
            float *Cb = Cs + (cc * kChunk + r0) * MS + r0 + j;
#pragma unroll
            for (int i2 = 0; i2 < kBlk; ++i2) Cb[i2 * MS] = x[i2];
        }
        __syncthreads();
        // the previous head's W store must have left the A tile before step 3 rewrites it (the
        // barriers inside the off-diagonal step order this wait before those writes)
        if (tid == 0) bulk_wait_read();
        if (hh == 0) {  // the event index of the group's chunks: the compaction's output
            pdl_wait();
            if (tid < 2) ev_s[tid] = (a.ev_of && tid < nch) ? a.ev_of[((int64_t)b * a.P_ + p) * a.C + c0 + tid] : -1;
        }
        offdiag_blocks<1>(Ms, Cs, Tb, tid);
        if (max_off == 3) {
            offdiag_blocks<2>(Ms, Cs, Tb, tid);
            offdiag_blocks<3>(Ms, Cs, Tb, tid);
        }
        const bool any_event = ev_s[0] >= 0 || ev_s[1] >= 0;  // published by the barriers above
        // 3. A tiles: C diag(beta) for U, and C diag(beta 2^g) for W (built in the
        //    fp32 M area, free once the solve is done); both bf16, block-diagonal
        {
            const float *crow = Cs + (ct * kChunk + tl) * MS;
            const int slab = seg >> 1, c0s = 32 * (seg & 1);  // this thread's 32 columns
            for (int part = 0; part < (any_event ? 2 : 1); ++part) {
                uint8_t *dst = (part == 0 ? sm + OFF_A : reinterpret_cast<uint8_t *>(Ms)) + slab * kSlab;
                const float *f = (part == 0 ? bet : bgs) + 64 * ct;
                if (slab == ct) {  // warp-uniform: these columns belong to the row's own chunk
#pragma unroll
                    for (int k0 = 0; k0 < 32; k0 += 8) {
                        // blocks the solver does not keep (and those above the diagonal) are zero
                        const int col = c0s + k0, jb = col >> 4, ib = tl >> 4;
                        float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        if (jb <= ib && (max_off == 3 || jb + 1 >= ib)) {
                            const float4 c0 = ld4(crow + col), c1 = ld4(crow + col + 4);
                            const float4 f0 = ld4(f + col), f1 = ld4(f + col + 4);
                            w[0] = c0.x * f0.x; w[1] = c0.y * f0.y; w[2] = c0.z * f0.z; w[3] = c0.w * f0.w;
                            w[4] = c1.x * f1.x; w[5] = c1.y * f1.y; w[6] = c1.z * f1.z; w[7] = c1.w * f1.w;
                        }
                        st_sw128_8(dst, row, col, w);
                    }
                } else {
                    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k0 = 0; k0 < 32; k0 += 8) st_sw128_8(dst, row, c0s + k0, z);
                }
            }
        }
        if (a.cbar) {  // compact C-bar = C diag(beta 2^g), bf16 as in the W operand, for the W kernel after selection
            for (int idx = tid; idx < nch * a.nblk * 32; idx += kThreads) {  // 8 coefficients (16 bytes) each
                const int cc = idx / (a.nblk * 32), rem = idx % (a.nblk * 32);
                const int blk = rem >> 5, rr = (rem >> 1) & 15, col0 = (rem & 1) * 8;
                const int rw = blk_row(blk) * kBlk + rr, cl = blk_col(blk) * kBlk + col0;
                const float *cr = Cs + (cc * kChunk + rw) * MS + cl;
                const float *bg = bgs + 64 * cc + cl;
                alignas(16) __nv_bfloat162 p2[4];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2)
                    p2[q2] = __floats2bfloat162_rn(cr[2 * q2] * bg[2 * q2], cr[2 * q2 + 1] * bg[2 * q2 + 1]);
                *reinterpret_cast<uint4 *>(a.cbar + (((int64_t)b * a.Nv + h) * a.C + c0 + cc) * a.nblk * 256 +
                                           blk * 256 + rr * 16 + col0) = *reinterpret_cast<uint4 *>(p2);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // 4. U = (C diag(beta)) V and, for events, W = (C diag(beta 2^g)) K
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, false, true);
            uint8_t *vt = sm + OFF_V + hh * 2 * kSlab;
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tbase + TM_U, kmajor_desc(smem_addr(sm + OFF_A), ks, kSlab),
                         mnmajor_desc(smem_addr(vt), ks, kSlab), id, ks > 0);
            mma_commit(&bar_u);
            if (any_event) {  // W on its own barrier: the U epilogue below overlaps it
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_W, kmajor_desc(smem_addr(Ms), ks, kSlab),
                             mnmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id, ks > 0);
                mma_commit(&bar_w);
            }
        }
        if (!mbar_wait(&bar_u, hh)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
        tc_fence_after();
        {   // U rows staged in this head's V tile (free once the MMAs are done), W rows in the A tile
            float sq = 0.f;
            const int slab = seg >> 1, c0s = 32 * (seg & 1);
            uint8_t *ustage = sm + OFF_V + hh * 2 * kSlab + slab * kSlab;
            {
                float u[32];
                tmem_ld32(tmem_addr(tbase, quarter * 32, TM_U + 32 * seg), u);
                tmem_ld_wait();
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(ustage, row, c0s + 8 * v8, &u[8 * v8]);
                if (in_tail) {
#pragma unroll
                    for (int q2 = 0; q2 < 32; ++q2) sq += u[q2] * u[q2];
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            if (lane == 0 && sq != 0.f) atomicAdd(&ssum[ct], sq);
            if (any_event && !mbar_wait(&bar_w, hh)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
            tc_fence_after();
            if (ev_s[ct] >= 0) {
                uint8_t *wstage = sm + OFF_A + slab * kSlab;
                float w[32];
                tmem_ld32(tmem_addr(tbase, quarter * 32, TM_W + 32 * seg), w);
                tmem_ld_wait();
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(wstage, row, c0s + 8 * v8, &w[8 * v8]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            uint8_t *ust = sm + OFF_V + hh * 2 * kSlab;
            tma_store_4d(&tU, 0, h, t0, b, ust);  // rows past the sequence's end are clipped
            tma_store_4d(&tU, 64, h, t0, b, ust + kSlab);
            for (int cc = 0; cc < nch; ++cc) {
                const int ev = ev_s[cc];
                if (ev < 0) continue;
                const int wrow = (ev * 2 + hh) * kChunk;
                tma_store_3d(&tW, 0, wrow, 0, sm + OFF_A + cc * 8192);
                tma_store_3d(&tW, 64, wrow, 0, sm + OFF_A + kSlab + cc * 8192);
            }
            bulk_commit();
        }
        tc_fence_before();
        __syncthreads();
        if (tid < nch && a.score) a.score[((int64_t)b * a.Nv + h) * a.C + c0 + tid] = sqrtf(ssum[tid]);
        __syncthreads();
    }
    if (tid == 0) bulk_wait_read();  // the stores only need their shared-memory sources before exit
    if (abort_s && tid == 0) {
        mbar_wait(&bar_ld, 0);
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    pdl_wait();  // also on an early exit: this grid's completion implies its predecessors'
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tbase);
}

}  // namespace

cudaError_t launch_intra_tc(const Problem &pb, const Workspace &ws, bool write_cbar) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tK, tV, tU, tW;
    const uint64_t wrows = (uint64_t)ws.ev_cap * 2 * kChunk;
    if (!make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tV, pb.v, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tU, ws.U, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_bf16_3d(&tW, ws.W, kDim, wrows, 1, kDim * 2, wrows * kDim * 2, 64, 64, 1))
        return cudaErrorInvalidValue;
    IntraParams a;
    a.beta = pb.beta; a.g = pb.g; a.ev_of = write_cbar ? nullptr : ws.ev_of;
    a.cbar = write_cbar ? reinterpret_cast<__nv_bfloat16 *>(ws.cbar) : nullptr;
    a.U = (__nv_bfloat16 *)ws.U; a.W = (__nv_bfloat16 *)ws.W; a.score = pb.score;
    a.status = ws.counts + 2;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.nblk = pb.nblk;
    a.exact = pb.solver == GDN_SOLVER_EXACT;
    a.tail = pb.tail;
    cudaFuncSetAttribute(intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraTcSmem);
    return launch_kernel(pb.pdl, intra_tc_kernel, dim3(pb.G, pb.P, pb.B), kThreads, kIntraTcSmem, pb.stream, tK, tV,
                         tU, tW, a);
}

}  // namespace gdn
