// k_scan.cu -- deferred W (SparseGDN Sec. 2.5, Eq. 15) and the event-sparse
// state scan (Sec. 2.6, Eqs. 17-21).
//
// wbuild_kernel: for every selected event e (chunk c of head pair p) and both
// value heads of the pair, W = C-bar_c K_c from the compact blocks:
//   W_0 = Cb_00 K_0,  W_i = Cb_ii K_i + Cb_i,i-1 K_i-1 (+ far blocks, exact solver).
// The event count E is read on the device; CTAs past E exit.
//
// scan_kernel: one CTA per (CSR row, value head of the pair, 32-column slice
// of dv).  Columns of S evolve independently (U'[:,v] and S[:,v] only read
// column v), so the state slice S[:, v0:v0+32] stays resident in shared
// memory while the CTA walks its row's events in time order:
//   S <- 2^(P_c - P_cur) S                     (gap decay over skipped chunks, Eq. 21)
//   U' = U_c - W_e S;  U_c <- U' in place      (Eq. 1)
//   S <- 2^gamma_c S + K_c^T (U' * 2^(gamma_c - g_c))   (Eq. 2)
//   snapshot S if a later output group reads this event
// and finally S_final = 2^(P_C - P_cur) S.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 32;   // dv columns per scan CTA

__device__ __forceinline__ int find_row(const int32_t *row_ptr, int R, int e) {
    // largest j with row_ptr[j] <= e (rows may be empty)
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (row_ptr[mid] <= e) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
wbuild_kernel(const T *__restrict__ K, const float *__restrict__ cbar, const int32_t *__restrict__ counts,
              const int32_t *__restrict__ row_pair, const int32_t *__restrict__ row_ptr,
              const int32_t *__restrict__ ev_chunk, int R, int P, int T_, int Nq, int Nv, int C, int nblk,
              int64_t ev_cap, T *__restrict__ W) {
    __shared__ float Ks[kChunk * kDim];
    __shared__ float Cb[kChunk * kChunk];  // dense 64x64 C-bar (stride 64: rows are read warp-uniformly)
    const int64_t E = min((int64_t)counts[0], ev_cap);
    const int tid = threadIdx.x;
    for (int64_t e = blockIdx.x; e < E; e += gridDim.x) {
        const int j = find_row(row_ptr, R, (int)e);
        const int i = row_pair[j], b = i / P, p = i % P, c = ev_chunk[e];
        const int64_t tok0 = (int64_t)b * T_ + (int64_t)c * kChunk;
        const int n = min(kChunk, T_ - c * kChunk);  // valid tokens (a partial last chunk has fewer)
        __syncthreads();
        for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
            const int t = idx / kDim, m = idx % kDim;
            Ks[idx] = t < n ? io<T>::ld(K + ((tok0 + t) * Nq + p) * kDim + m) : 0.f;
        }
        for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * p + hh;
            for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Cb[idx] = 0.f;
            __syncthreads();
            const float *cb = cbar + (((int64_t)b * Nv + h) * C + c) * nblk * 256;
            for (int idx = tid; idx < nblk * 256; idx += kThreads) {
                const int blk = idx >> 8, r = (idx >> 4) & 15, col = idx & 15;
                Cb[(blk_row(blk) * kBlk + r) * kChunk + blk_col(blk) * kBlk + col] = cb[idx];
            }
            __syncthreads();
            const int ty = tid >> 5, tx = tid & 31;
            float acc[8][4];
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[a][q] = 0.f;
            for (int s = 0; s < ty * 8 + 8; ++s) {
                float kv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) kv[q] = Ks[s * kDim + tx + 32 * q];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const float cf = Cb[(ty * 8 + a) * kChunk + s];
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] += cf * kv[q];
                }
            }
            T *w = W + ((e * 2 + hh) * kChunk) * kDim;
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) io<T>::st(w + (ty * 8 + a) * kDim + tx + 32 * q, acc[a][q]);
            __syncthreads();
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
scan_kernel(const T *__restrict__ K, const T *__restrict__ W, T *__restrict__ U, const float *__restrict__ g,
            const float *__restrict__ h0, const double *__restrict__ Pfx, const int32_t *__restrict__ counts,
            const int32_t *__restrict__ row_pair, const int32_t *__restrict__ row_ptr,
            const int32_t *__restrict__ ev_chunk, const int32_t *__restrict__ snap_slot,
            int P, int T_, int Nq, int Nv, int C, int64_t ev_cap, int64_t snap_cap,
            float *__restrict__ snap, float *__restrict__ s_final) {
    extern __shared__ float sm[];
    float *Ss = sm;                         // [128][32] state slice
    float *Ws = Ss + kDim * kSlice;         // [64][132]
    float *Ks = Ws + kChunk * (kDim + 4);   // [64][128]
    float *Us = Ks + kChunk * kDim;         // [64][33]
    float *gg = Us + kChunk * (kSlice + 1); // [64]
    const int j = blockIdx.x, hh = blockIdx.y, v0 = blockIdx.z * kSlice, tid = threadIdx.x;
    const int i = row_pair[j], b = i / P, p = i % P, h = 2 * p + hh;
    const double *Pu = Pfx + ((int64_t)b * Nv + h) * (C + 1);
    const int64_t sbase = ((int64_t)b * Nv + h) * kDim * kDim;

    // thread ownership of the slice: rows m = tid/2, columns (tid&1)*16 + q
    const int sm_row = tid >> 1, sm_col = (tid & 1) * 16;
    for (int q = 0; q < 16; ++q)
        Ss[sm_row * kSlice + sm_col + q] = h0 ? h0[sbase + (int64_t)sm_row * kDim + v0 + sm_col + q] : 0.f;

    const int64_t e_beg = min((int64_t)row_ptr[j], ev_cap), e_end = min((int64_t)row_ptr[j + 1], ev_cap);
    int cur = 0;
    for (int64_t e = e_beg; e < e_end; ++e) {
        const int c = ev_chunk[e];
        const int64_t tok0 = (int64_t)b * T_ + (int64_t)c * kChunk;
        const int n = min(kChunk, T_ - c * kChunk);  // valid tokens (a partial last chunk has fewer)
        __syncthreads();
        const T *w = W + (e * 2 + hh) * kChunk * kDim;
        for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
            const int t = idx / kDim, m = idx % kDim;
            Ws[t * (kDim + 4) + m] = io<T>::ld(w + idx);
            Ks[idx] = t < n ? io<T>::ld(K + ((tok0 + t) * Nq + p) * kDim + m) : 0.f;
        }
        for (int idx = tid; idx < kChunk * kSlice; idx += kThreads) {
            const int t = idx / kSlice, v = idx % kSlice;
            Us[t * (kSlice + 1) + v] = t < n ? io<T>::ld(U + ((tok0 + t) * Nv + h) * kDim + v0 + v) : 0.f;
        }
        if (tid < kChunk) gg[tid] = g[(tok0 + min(tid, n - 1)) * Nv + h];  // gg[63]: g at the last token
        const float gap = exp2f((float)(Pu[c] - Pu[cur]));
        for (int q = 0; q < 16; ++q) Ss[sm_row * kSlice + sm_col + q] *= gap;
        __syncthreads();
        const float gam = gg[kChunk - 1];
        {   // U' = U - W S ; write back in place; keep U' 2^(gamma - g) for the state write
            const int t = tid >> 2;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.f;
            for (int m = 0; m < kDim; ++m) {
                const float wv = Ws[t * (kDim + 4) + m];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += wv * Ss[m * kSlice + (tid & 3) + 4 * q];
            }
            const float dec = exp2f(gam - gg[t]);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int v = (tid & 3) + 4 * q;
                const float up = Us[t * (kSlice + 1) + v] - acc[q];
                if (t < n) io<T>::st(U + ((tok0 + t) * Nv + h) * kDim + v0 + v, up);
                Us[t * (kSlice + 1) + v] = up * dec;
            }
        }
        __syncthreads();
        {   // S <- 2^gamma S + K^T (U' 2^(gamma-g))
            const float dg = exp2f(gam);
            float acc[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[q] = 0.f;
            for (int t = 0; t < kChunk; ++t) {
                const float kv = Ks[t * kDim + sm_row];
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] += kv * Us[t * (kSlice + 1) + sm_col + q];
            }
            const int slot = snap_slot[e];
            const bool keep = slot >= 0 && slot < snap_cap;
            float *sn = snap + (((int64_t)slot * 2 + hh) * kDim + sm_row) * kDim + v0 + sm_col;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float s = dg * Ss[sm_row * kSlice + sm_col + q] + acc[q];
                Ss[sm_row * kSlice + sm_col + q] = s;
                if (keep) sn[q] = s;
            }
        }
        cur = c + 1;
    }
    const float tail = exp2f((float)(Pu[C] - Pu[cur]));
    for (int q = 0; q < 16; ++q)
        s_final[sbase + (int64_t)sm_row * kDim + v0 + sm_col + q] = tail * Ss[sm_row * kSlice + sm_col + q];
}

constexpr size_t kScanSmem =
    sizeof(float) * (kDim * kSlice + kChunk * (kDim + 4) + kChunk * kDim + kChunk * (kSlice + 1) + kChunk);

}  // namespace

cudaError_t launch_wbuild(const Problem &pb, const Workspace &ws) {
    if (pb.R == 0 || pb.C == 0) return cudaSuccess;
    const int grid = (int)(ws.ev_cap < 152 * 8 ? ws.ev_cap : 152 * 8);
    if (pb.dtype == GDN_BF16)
        wbuild_kernel<__nv_bfloat16><<<grid, kThreads, 0, pb.stream>>>(
            (const __nv_bfloat16 *)pb.k, ws.cbar, ws.counts, ws.row_pair, ws.row_ptr, ws.ev_chunk, pb.R, pb.P, pb.T,
            pb.Nq, pb.Nv, pb.C, pb.nblk, ws.ev_cap, (__nv_bfloat16 *)ws.W);
    else
        wbuild_kernel<float><<<grid, kThreads, 0, pb.stream>>>(
            (const float *)pb.k, ws.cbar, ws.counts, ws.row_pair, ws.row_ptr, ws.ev_chunk, pb.R, pb.P, pb.T, pb.Nq,
            pb.Nv, pb.C, pb.nblk, ws.ev_cap, (float *)ws.W);
    return cudaGetLastError();
}

cudaError_t launch_scan(const Problem &pb, const Workspace &ws) {
    if (pb.R == 0) return cudaSuccess;
    dim3 grid(pb.R, 2, kDim / kSlice);
    if (pb.dtype == GDN_BF16) {
        auto kern = scan_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
        kern<<<grid, kThreads, kScanSmem, pb.stream>>>(
            (const __nv_bfloat16 *)pb.k, (const __nv_bfloat16 *)ws.W, (__nv_bfloat16 *)ws.U, pb.g, pb.h0, ws.P,
            ws.counts, ws.row_pair, ws.row_ptr, ws.ev_chunk, ws.snap_slot, pb.P, pb.T, pb.Nq, pb.Nv, pb.C, ws.ev_cap,
            ws.snap_cap, (float *)ws.snap, pb.s_final);
    } else {
        auto kern = scan_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
        kern<<<grid, kThreads, kScanSmem, pb.stream>>>(
            (const float *)pb.k, (const float *)ws.W, (float *)ws.U, pb.g, pb.h0, ws.P, ws.counts, ws.row_pair,
            ws.row_ptr, ws.ev_chunk, ws.snap_slot, pb.P, pb.T, pb.Nq, pb.Nv, pb.C, ws.ev_cap, ws.snap_cap, (float *)ws.snap,
            pb.s_final);
    }
    return cudaGetLastError();
}

}  // namespace gdn
