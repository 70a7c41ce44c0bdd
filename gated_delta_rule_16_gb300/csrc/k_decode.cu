// k_decode.cu -- single-token decode step from the prefill's final state
// (SparseGDN Sec. 2.6: S_C is returned for the autoregressive decoding that
// follows; Eqs. 1-4 for a chunk of one token with log2 retention a, where
// g = gamma = a, A_Delta is empty and M = 1):
//   U' = beta v - beta 2^a S^T k,   S <- 2^a S + k U'^T,
//   o  = [2^a S^T q + <q,k> U'] / sqrt(d)      (= S_new^T q / sqrt(d))
//
// One CTA per (sequence, value head), 512 threads: thread (j, r) owns column j of
// S (a d_v index) for the 32 rows 32r .. 32r+31, held in registers between the two
// passes.  Each row of S is read and written by 128 consecutive threads (512
// contiguous bytes).  Memory-bound: 64 KiB read and 64 KiB written per head.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;

template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const float *__restrict__ beta, const float *__restrict__ a, float *__restrict__ state,
              T *__restrict__ o, int Nq, int Nv) {
    __shared__ float qs[kDim], ks[kDim], red_k[4][kDim], red_q[4][kDim], qk_s;
    const int bh = blockIdx.x, b = bh / Nv, h = bh % Nv, p = h / 2;
    const int tid = threadIdx.x, j = tid & (kDim - 1), r = tid >> 7;
    const int64_t qoff = ((int64_t)b * Nq + p) * kDim;
    if (tid < kDim) {
        qs[tid] = io<T>::ld(q + qoff + tid);
        ks[tid] = io<T>::ld(k + qoff + tid);
    }
    float *S = state + (int64_t)bh * kDim * kDim;
    float s_reg[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s_reg[i] = S[(int64_t)(32 * r + i) * kDim + j];
    __syncthreads();
    if (tid < 32) {  // <q, k>
        float x = 0.f;
        for (int i = tid; i < kDim; i += 32) x += qs[i] * ks[i];
#pragma unroll
        for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (tid == 0) qk_s = x;
    }
    float pk = 0.f, pq = 0.f;  // partial k^T S and q^T S of column j over this thread's rows
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        pk += ks[32 * r + i] * s_reg[i];
        pq += qs[32 * r + i] * s_reg[i];
    }
    red_k[r][j] = pk;
    red_q[r][j] = pq;
    __syncthreads();
    const float kS = red_k[0][j] + red_k[1][j] + red_k[2][j] + red_k[3][j];
    const float qS = red_q[0][j] + red_q[1][j] + red_q[2][j] + red_q[3][j];
    const float bt = beta[(int64_t)b * Nv + h], decay = exp2f(a[(int64_t)b * Nv + h]);
    const float up = bt * io<T>::ld(v + ((int64_t)b * Nv + h) * kDim + j) - bt * decay * kS;  // U'_j
#pragma unroll
    for (int i = 0; i < 32; ++i) S[(int64_t)(32 * r + i) * kDim + j] = decay * s_reg[i] + ks[32 * r + i] * up;
    if (r == 0)
        io<T>::st(o + ((int64_t)b * Nv + h) * kDim + j, (decay * qS + qk_s * up) * rsqrtf((float)kDim));
}

}  // namespace

cudaError_t launch_decode(const gdn_shape &s, const void *q, const void *k, const void *v, const float *beta,
                          const float *a, float *state, void *o, cudaStream_t stream) {
    if (s.B == 0) return cudaSuccess;
    const int grid = s.B * s.Nv;
    if (s.dtype == GDN_BF16)
        decode_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, beta, a, state,
            (__nv_bfloat16 *)o, s.Nq, s.Nv);
    else
        decode_kernel<float><<<grid, kThreads, 0, stream>>>((const float *)q, (const float *)k, (const float *)v,
                                                           beta, a, state, (float *)o, s.Nq, s.Nv);
    return cudaGetLastError();
}

}  // namespace gdn
