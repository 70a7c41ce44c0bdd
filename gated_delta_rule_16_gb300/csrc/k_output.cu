// k_output.cu -- mapped two-chunk group output (SparseGDN Sec. 2.7, Eqs. 22-24).
//
// One CTA per (group r, head pair p, sequence b); group r covers chunks
// c = 2r and c+1.  Per value head of the pair:
//   entry state S_c: the snapshot of the group's predecessor event e (the last
//   event with chunk < c), decayed over the gap, S_c = 2^(P_c - P_e+1) snap[e]
//   (Eq. 21); 2^P_c h0 when no event precedes the group (0 without h0).
//   O_c   = [2^g_c * (Q_c S_c) + A_cc U'_c] / sqrt(d)
//   O_c+1 = [2^(g_c+1 + gamma_c) * (Q_c+1 S_c) + A_c+1,c U'_c + A_c+1,c+1 U'_c+1] / sqrt(d)
//   A_cc[i,j]   = <q_i,k_j> 2^(g_i - g_j) [j <= i]
//   A_c+1,c[i,j] = <q_c+1,i, k_c,j> 2^(g_c+1,i + gamma_c - g_c,j)   (no mask)
// U' is read from the workspace U buffer, where the scan replaced U by U' for
// selected chunks.  All arithmetic fp32 on CUDA cores.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int QS_ = kDim + 1;
constexpr size_t kOutSmem = sizeof(float) * (kDim * kDim + 2 * kChunk * QS_ + kChunk * (kChunk + 1) +
                                             kChunk * kDim + 2 * kChunk);

template <typename T>
__global__ void __launch_bounds__(kThreads)
output_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ U,
              const float *__restrict__ g, const float *__restrict__ h0, const double *__restrict__ Pfx,
              const int32_t *__restrict__ ev_chunk, const int32_t *__restrict__ grp_pred,
              const int32_t *__restrict__ snap_slot, const float *__restrict__ snap, int P, int T_, int Nq,
              int Nv, int C, int G, int64_t ev_cap, int64_t snap_cap, T *__restrict__ O) {
    extern __shared__ float sm[];
    float *Ss = sm;                  // [128][128] entry state
    float *Qs = Ss + kDim * kDim;    // [64][129]
    float *Ks = Qs + kChunk * QS_;   // [64][129]
    float *As = Ks + kChunk * QS_;   // [64][65]
    float *Us = As + kChunk * (kChunk + 1); // [64][128]
    float *gq = Us + kChunk * kDim;  // [64]
    float *gk = gq + kChunk;         // [64]
    const int r = blockIdx.x, p = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int c0 = 2 * r, nparts = (c0 + 1 < C) ? 2 : 1;
    const int ty = tid >> 5, tx = tid & 31;
    const float inv_sqrt_d = rsqrtf((float)kDim);
    const int pred = grp_pred[((int64_t)b * P + p) * G + r];

    for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * p + hh;
        const double *Pu = Pfx + ((int64_t)b * Nv + h) * (C + 1);
        __syncthreads();
        // entry state of the group
        {
            const float *src = nullptr;
            float f = 0.f;
            if (pred >= 0 && pred < ev_cap) {
                const int slot = snap_slot[pred];
                if (slot >= 0 && slot < snap_cap) {
                    src = snap + ((int64_t)slot * 2 + hh) * kDim * kDim;
                    f = exp2f((float)(Pu[c0] - Pu[ev_chunk[pred] + 1]));
                }
            } else if (h0) {
                src = h0 + ((int64_t)b * Nv + h) * kDim * kDim;
                f = exp2f((float)Pu[c0]);
            }
            for (int idx = tid; idx < kDim * kDim; idx += kThreads) Ss[idx] = src ? f * src[idx] : 0.f;
        }
        for (int part = 0; part < nparts; ++part) {
            const int cq = c0 + part;
            const int64_t tq0 = (int64_t)b * T_ + (int64_t)cq * kChunk;
            const int nq = min(kChunk, T_ - cq * kChunk);  // valid query tokens (a partial last chunk has fewer)
            __syncthreads();
            for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
                const int t = idx / kDim, m = idx % kDim;
                Qs[t * QS_ + m] = t < nq ? io<T>::ld(Q + ((tq0 + t) * Nq + p) * kDim + m) : 0.f;
            }
            if (tid < kChunk) gq[tid] = g[(tq0 + min(tid, nq - 1)) * Nv + h];
            __syncthreads();
            const float shift = part ? g[((int64_t)b * T_ + (int64_t)c0 * kChunk + kChunk - 1) * Nv + h] : 0.f;
            float acc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            for (int m = 0; m < kDim; ++m) {
                float sv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) sv[j] = Ss[m * kDim + tx + 32 * j];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float qv = Qs[(ty * 8 + i) * QS_ + m];
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] += qv * sv[j];
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float f = exp2f(gq[ty * 8 + i] + shift);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] *= f;
            }
            // local terms: part 0 -> (c0, causal); part 1 -> (c0, cross) and (c0+1, causal)
            for (int term = 0; term <= part; ++term) {
                const int ck = c0 + term;
                const bool cross = part == 1 && term == 0;
                const int64_t tk0 = (int64_t)b * T_ + (int64_t)ck * kChunk;
                const int nk = min(kChunk, T_ - ck * kChunk);
                __syncthreads();
                for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
                    const int t = idx / kDim, m = idx % kDim;
                    Ks[t * QS_ + m] = t < nk ? io<T>::ld(K + ((tk0 + t) * Nq + p) * kDim + m) : 0.f;
                    Us[idx] = t < nk ? io<T>::ld(U + ((tk0 + t) * Nv + h) * kDim + m) : 0.f;
                }
                if (tid < kChunk) gk[tid] = g[(tk0 + min(tid, nk - 1)) * Nv + h];
                __syncthreads();
                {   // A tile: row t = tid/4, columns s = tid%4 + 4j
                    const int t = tid >> 2;
                    float a[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = 0.f;
                    for (int m = 0; m < kDim; ++m) {
                        const float qv = Qs[t * QS_ + m];
#pragma unroll
                        for (int j = 0; j < 16; ++j) a[j] += qv * Ks[((tid & 3) + 4 * j) * QS_ + m];
                    }
                    const float gam_k = gk[kChunk - 1];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = (tid & 3) + 4 * j;
                        float w;
                        if (cross) w = exp2f(gq[t] + gam_k - gk[s]);
                        else w = s <= t ? exp2f(gq[t] - gk[s]) : 0.f;
                        As[t * (kChunk + 1) + s] = a[j] * w;
                    }
                }
                __syncthreads();
                const int smax = cross ? kChunk : ty * 8 + 8;
                for (int s = 0; s < smax; ++s) {
                    float uv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) uv[j] = Us[s * kDim + tx + 32 * j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float av = As[(ty * 8 + i) * (kChunk + 1) + s];
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] += av * uv[j];
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (ty * 8 + i < nq)
                        io<T>::st(O + ((tq0 + ty * 8 + i) * Nv + h) * kDim + tx + 32 * j, acc[i][j] * inv_sqrt_d);
        }
    }
}

}  // namespace

cudaError_t launch_output(const Problem &pb, const Workspace &ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    dim3 grid(pb.G, pb.P, pb.B);
    if (pb.dtype == GDN_BF16) {
        auto kern = output_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem);
        kern<<<grid, kThreads, kOutSmem, pb.stream>>>(
            (const __nv_bfloat16 *)pb.q, (const __nv_bfloat16 *)pb.k, (const __nv_bfloat16 *)ws.U, pb.g, pb.h0, ws.P,
            ws.ev_chunk, ws.grp_pred, ws.snap_slot, (float *)ws.snap, pb.P, pb.T, pb.Nq, pb.Nv, pb.C, pb.G, ws.ev_cap,
            ws.snap_cap, (__nv_bfloat16 *)pb.o);
    } else {
        auto kern = output_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem);
        kern<<<grid, kThreads, kOutSmem, pb.stream>>>(
            (const float *)pb.q, (const float *)pb.k, (const float *)ws.U, pb.g, pb.h0, ws.P, ws.ev_chunk,
            ws.grp_pred, ws.snap_slot, (float *)ws.snap, pb.P, pb.T, pb.Nq, pb.Nv, pb.C, pb.G, ws.ev_cap, ws.snap_cap,
            (float *)pb.o);
    }
    return cudaGetLastError();
}

}  // namespace gdn
