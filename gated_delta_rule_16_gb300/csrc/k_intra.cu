// k_intra.cu -- intra-chunk step (SparseGDN Sec. 2.3, Eqs. 5-9) and the
// per-head log2 decay prefix P (Sec. 2.6, Eq. 19).
//
// intra_kernel: one CTA per (chunk c, head pair p, sequence b).  The pair's two
// value heads share the key Gram matrix K_c K_c^T, formed once.  Per head:
//   A_Delta[t,s] = beta_t <k_t,k_s> 2^(g_t - g_s)   (s < t),  M = I + A_Delta
//   C = M^-1 (exact) or its block-adjacent approximation (Eq. 7):
//       C_ii = M_ii^-1,  C_ij = -C_ii sum_{k=j}^{i-1} M_ik C_kj
//       (offsets i-j = 1 only for the block-adjacent solver, 1..3 for exact)
//   U = C diag(beta) V               -> workspace U  [B,T,Nv,dv] (dtype)
//   C-bar = C diag(beta 2^g)         -> compact blocks [B,Nv,C,nblk,16,16] fp32
//   s = ||U[48:64,:]||_F             -> score [B,Nv,C] (Tail-16 write score)
// All arithmetic is fp32 on CUDA cores.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int KS = kChunk * (kDim + 1);   // K tile, row stride 129
constexpr int MS = kChunk * (kChunk + 1); // 64x64 tiles, row stride 65
constexpr int VS = kChunk * kDim;         // V / U tile, row stride 128
constexpr size_t kIntraSmem = sizeof(float) * (KS + 3 * MS + VS + 3 * 256 + 2 * kChunk + 8);

template <typename T>
__global__ void __launch_bounds__(kThreads)
intra_kernel(const T *__restrict__ K, const T *__restrict__ V, const float *__restrict__ beta,
             const float *__restrict__ g, int T_, int Nq, int Nv, int C, int nblk, int exact, int tail,
             T *__restrict__ U, float *__restrict__ cbar, float *__restrict__ score) {
    extern __shared__ float sm[];
    float *Ks = sm;            // [64][129]
    float *Gs = Ks + KS;       // [64][65]  K K^T
    float *Ms = Gs + MS;       // [64][65]  M
    float *Cs = Ms + MS;       // [64][65]  C
    float *Vs = Cs + MS;       // [64][128]
    float *Tb = Vs + VS;       // [3][16][16]
    float *bet = Tb + 3 * 256; // [64]
    float *gg = bet + kChunk;  // [64]
    float *red = gg + kChunk;  // [8]
    const int c = blockIdx.x, p = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int64_t tok0 = (int64_t)b * T_ + (int64_t)c * kChunk;
    const int n = min(kChunk, T_ - c * kChunk);  // valid tokens (a partial last chunk has fewer)

    for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
        const int t = idx / kDim, m = idx % kDim;
        Ks[t * (kDim + 1) + m] = t < n ? io<T>::ld(K + ((tok0 + t) * Nq + p) * kDim + m) : 0.f;
    }
    __syncthreads();
    {   // Gram matrix: thread owns row t, columns s = tid%4 + 4j
        const int t = tid >> 2;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int m = 0; m < kDim; ++m) {
            const float a = Ks[t * (kDim + 1) + m];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] += a * Ks[((tid & 3) + 4 * j) * (kDim + 1) + m];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) Gs[t * (kChunk + 1) + (tid & 3) + 4 * j] = acc[j];
    }
    __syncthreads();

    for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * p + hh;
        if (tid < kChunk) {  // past the sequence's end: beta = 0 and a finite g
            bet[tid] = tid < n ? beta[(tok0 + tid) * Nv + h] : 0.f;
            gg[tid] = g[(tok0 + min(tid, n - 1)) * Nv + h];
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
            const int t = idx >> 6, s = idx & 63;
            float m = 0.f;
            if (s < t) m = bet[t] * Gs[t * (kChunk + 1) + s] * exp2f(gg[t] - gg[s]);
            else if (s == t) m = 1.f;
            Ms[t * (kChunk + 1) + s] = m;
            Cs[t * (kChunk + 1) + s] = 0.f;
        }
        __syncthreads();
        // diagonal blocks: forward substitution, one thread per (block, column)
        if (tid < kChunk) {
            const int j = tid, r1 = (j & ~15) + kBlk;
            Cs[j * (kChunk + 1) + j] = 1.f;
            for (int i = j + 1; i < r1; ++i) {
                float acc = 0.f;
                for (int s = j; s < i; ++s) acc += Ms[i * (kChunk + 1) + s] * Cs[s * (kChunk + 1) + j];
                Cs[i * (kChunk + 1) + j] = -acc;
            }
        }
        __syncthreads();
        // off-diagonal blocks by increasing distance
        const int max_off = exact ? 3 : 1;
        for (int off = 1; off <= max_off; ++off) {
            const int nb = 4 - off;
            for (int idx = tid; idx < nb * 256; idx += kThreads) {
                const int bi = idx >> 8, r = (idx >> 4) & 15, col = idx & 15;
                const int i = bi + off, j = bi;
                float acc = 0.f;  // (sum_k M_ik C_kj)[r, col]
                for (int kk = j * kBlk; kk < i * kBlk; ++kk)
                    acc += Ms[(i * kBlk + r) * (kChunk + 1) + kk] * Cs[kk * (kChunk + 1) + j * kBlk + col];
                Tb[idx] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < nb * 256; idx += kThreads) {
                const int bi = idx >> 8, r = (idx >> 4) & 15, col = idx & 15;
                const int i = bi + off, j = bi;
                float acc = 0.f;
                for (int m = 0; m < kBlk; ++m)
                    acc += Cs[(i * kBlk + r) * (kChunk + 1) + i * kBlk + m] * Tb[(bi << 8) + m * 16 + col];
                Cs[(i * kBlk + r) * (kChunk + 1) + j * kBlk + col] = -acc;
            }
            __syncthreads();
        }
        // compact C-bar = C diag(beta 2^g)
        float *cb = cbar + (((int64_t)b * Nv + h) * C + c) * nblk * 256;
        for (int idx = tid; idx < nblk * 256; idx += kThreads) {
            const int blk = idx >> 8, r = (idx >> 4) & 15, col = idx & 15;
            const int row = blk_row(blk) * kBlk + r, cl = blk_col(blk) * kBlk + col;
            cb[idx] = Cs[row * (kChunk + 1) + cl] * bet[cl] * exp2f(gg[cl]);
        }
        for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
            const int t = idx / kDim, m = idx % kDim;
            Vs[idx] = t < n ? io<T>::ld(V + ((tok0 + t) * Nv + h) * kDim + m) * bet[t] : 0.f;
        }
        __syncthreads();
        // U = C (diag(beta) V): thread rows ty*8+i, columns tx+32j
        const int ty = tid >> 5, tx = tid & 31;
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        const int smax = ty * 8 + 8;
        for (int s = 0; s < smax; ++s) {
            float bv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Vs[s * kDim + tx + 32 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float a = Cs[(ty * 8 + i) * (kChunk + 1) + s];
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] += a * bv[j];
            }
        }
        float sq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = ty * 8 + i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (t < n) io<T>::st(U + ((tok0 + t) * Nv + h) * kDim + tx + 32 * j, acc[i][j]);
                if (t >= n - tail && t < n) sq += acc[i][j] * acc[i][j];  // Tail-W: the last W valid rows
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (tx == 0) red[ty] = sq;
        __syncthreads();
        if (tid == 0 && score) {
            float s = 0.f;
            for (int w = 0; w < 8; ++w) s += red[w];
            score[((int64_t)b * Nv + h) * C + c] = sqrtf(s);
        }
        __syncthreads();
    }
}

// P[b,h,0] = 0, P[b,h,c+1] = P[b,h,c] + gamma_c (Eq. 19), fp64: one CTA per
// (sequence, head pair), one warp per value head.  Then, per output group r of
// the pair, the entry-state table the group output reads with one load:
// {snapshot slot or -1, state kind, 2^(P_2r - P_(e+1)) of both heads} where e is
// the group's predecessor event (kind 1), or {-1, 2, 2^P_2r} when the group
// starts from h0 (kind 2), or kind 0 (zero state).
__global__ void __launch_bounds__(256)
prefix_kernel(const float *__restrict__ g, int T_, int Nv, int C, int P_, int G,
              const int32_t *__restrict__ grp_pred, const int32_t *__restrict__ snap_slot,
              const int32_t *__restrict__ ev_chunk, int64_t ev_cap, int64_t snap_cap, int has_h0,
              double *__restrict__ P, int4 *__restrict__ grp_info, int p_in_smem) {
    extern __shared__ double Ps[];  // [2][C + 1]: P of both heads, for the group table (when it fits)
    const int bp = blockIdx.x, b = bp / P_, p = bp % P_;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    if (warp < 2) {  // P needs only the gates: it overlaps the kernel before  // warp hh scans head 2p + hh: the gate tails of 32 chunks per step, loads issued ahead
        const int h = 2 * p + warp;
        double *Pu = P + ((int64_t)b * Nv + h) * (C + 1);
        double *Pl = p_in_smem ? Ps + warp * (C + 1) : Pu;
        if (lane == 0) { Pu[0] = 0.0; Pl[0] = 0.0; }
        double carry = 0.0;
        for (int c0 = 0; c0 < C; c0 += 256) {
            double x[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + 32 * q + lane;
                // gamma_c: g at the chunk's last token (a partial last chunk ends at T - 1)
                x[q] = c < C ? (double)g[((int64_t)b * T_ + min((int64_t)c * kChunk + kChunk, (int64_t)T_) - 1) * Nv + h] : 0.0;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                double v = x[q];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += y;
                }
                const int c = c0 + 32 * q + lane;
                if (c < C) { Pu[c + 1] = carry + v; Pl[c + 1] = carry + v; }
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
        }
    }
    pdl_wait();  // the group table reads the compaction's output
    if (!grp_info) return;
    __syncthreads();  // P of both heads written (shared memory, or global memory by this CTA)
    const double *P0 = p_in_smem ? Ps : P + ((int64_t)b * Nv + 2 * p) * (C + 1);
    const double *P1 = P0 + (C + 1);
    for (int r = threadIdx.x; r < G; r += blockDim.x) {
        const int pred = grp_pred[(int64_t)bp * G + r];
        int4 info = make_int4(-1, 0, 0, 0);
        if (pred >= 0 && pred < ev_cap) {
            const int slot = snap_slot[pred];
            if (slot >= 0 && slot < snap_cap) {
                const int e1 = ev_chunk[pred] + 1;
                info = make_int4(slot, 1, __float_as_int(exp2f((float)(P0[2 * r] - P0[e1]))),
                                 __float_as_int(exp2f((float)(P1[2 * r] - P1[e1]))));
            }
        } else if (has_h0) {
            info = make_int4(-1, 2, __float_as_int(exp2f((float)P0[2 * r])), __float_as_int(exp2f((float)P1[2 * r])));
        }
        grp_info[(int64_t)bp * G + r] = info;
    }
}

}  // namespace

cudaError_t launch_intra(const Problem &pb, const Workspace &ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    dim3 grid(pb.C, pb.P, pb.B);
    const int exact = pb.solver == GDN_SOLVER_EXACT;
    if (pb.dtype == GDN_BF16) {
        auto kern = intra_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraSmem);
        kern<<<grid, kThreads, kIntraSmem, pb.stream>>>(
            (const __nv_bfloat16 *)pb.k, (const __nv_bfloat16 *)pb.v, pb.beta, pb.g, pb.T, pb.Nq, pb.Nv, pb.C,
            pb.nblk, exact, pb.tail, (__nv_bfloat16 *)ws.U, ws.cbar, pb.score);
    } else {
        auto kern = intra_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraSmem);
        kern<<<grid, kThreads, kIntraSmem, pb.stream>>>(
            (const float *)pb.k, (const float *)pb.v, pb.beta, pb.g, pb.T, pb.Nq, pb.Nv, pb.C, pb.nblk, exact, pb.tail,
            (float *)ws.U, ws.cbar, pb.score);
    }
    return cudaGetLastError();
}

cudaError_t launch_prefix(const Problem &pb, const Workspace &ws) {
    if (pb.R == 0) return cudaSuccess;
    const size_t want = 2 * (size_t)(pb.C + 1) * sizeof(double);
    const int in_smem = want <= 96 * 1024;  // else the group table reads P from global memory
    const size_t smem = in_smem ? want : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(pb.pdl, prefix_kernel, pb.R, 256, smem, pb.stream, pb.g, pb.T, pb.Nv, pb.C, pb.P, pb.G,
                         (const int32_t *)ws.grp_pred, (const int32_t *)ws.snap_slot, (const int32_t *)ws.ev_chunk,
                         ws.ev_cap, ws.snap_cap, (int)(pb.h0 != nullptr), ws.P, (int4 *)ws.grp_info, in_smem);
}

}  // namespace gdn
