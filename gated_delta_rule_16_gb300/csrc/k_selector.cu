// k_selector.cu -- online event selection (SparseGDN Sec. 2.4, Eqs. 10-14).
//
// Two kernels: one CTA per (head pair, sequence) ranks the pair's chunks and sums its
// upgrade gains; one CTA per sequence then picks the tiers (16 head pairs, the pages'
// tier table) and writes the mask.  From the Tail-16
// scores s[h][c] of the intra step, the chunk gate tails gamma (read from g at
// each chunk's last token) and an optional output-visibility energy eta[h]:
//   norm_h = ||s_{.,h}||_2            fp64 sum of squares, rounded to fp32, fp32 sqrt
//   q_c    = 0.5 (s_{c,h0}/norm_h0 + s_{c,h1}/norm_h1)   fp32, IEEE division (Eq. 10)
//   r_h    = mean 2^gamma over the last min(16, C) chunks; L_h = sum_{j=1}^{C-2} r_h^j (Eq. 11)
//   G_h    = sqrt(eta_h / mean eta) or 1                  (Eq. 11)
//   k_l    = clip(round_half_even(rho_l C), 2, C), rho = (0.08, 0.30, 0.95)
//   C_l    = anchors {0, C-1} + the k_l - 2 best non-anchor chunks by q (ties: lower chunk)
//   gains  = sum over C_b \ C_a of s L G (Eq. 12), fp64; x = gains / mean over pairs
//   n_H    = argmax_{1..4} B(x_H), n_M = argmax over the table row of B(x_M of the rest) (Eq. 14)
// The ranking of each pair is a bitonic sort in shared memory of 64-bit keys
// (~bits(q) << 32 | chunk), i.e. q descending then chunk ascending (q >= 0: the
// scores are norms); q is computed with IEEE fp32 division from the fp32 norms,
// as in the sequential definition.  The fp64 quantities behind the tier choice
// (sums of squares, L_h, gains, separations) are reduced in parallel: they
// differ from a sequential evaluation only in rounding order (and exp2's last
// ulp), so a tier choice can only differ where two candidates are within fp64
// rounding of each other.  GB300's fp64 units are slow (a dependent fp64 add
// costs on the order of a hundred cycles), so no step here is a long serial chain.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;
constexpr int kPairs = 16;

// B(x, k) of Eq. 14 for sorted x[0..n): k (n - k) / n (mean of the top k - mean of the rest)^2
__device__ double separation(const double *xs, int n, int k) {
    double top = 0.0, rest = 0.0;
    for (int i = 0; i < k; ++i) top += xs[i];
    for (int i = k; i < n; ++i) rest += xs[i];
    top /= k;
    rest = n > k ? rest / (n - k) : 0.0;
    return (double)k * (n - k) / n * (top - rest) * (top - rest);
}

// position of element i in x sorted descending, ties to the lower index
__device__ __forceinline__ int desc_position(const double *x, const int *ids, int n, int i) {
    const double v = x[ids[i]];
    int pos = 0;
    for (int j = 0; j < n; ++j) {
        const double u = x[ids[j]];
        pos += (u > v || (u == v && ids[j] < ids[i])) ? 1 : 0;
    }
    return pos;
}

// x^n for n >= 1 by binary exponentiation (a short dependent chain: fp64 is slow here)
__device__ __forceinline__ double ipow(double x, int n) {
    double r = 1.0;
    while (n) {
        if (n & 1) r *= x;
        x *= x;
        n >>= 1;
    }
    return r;
}

template <int NT>
__device__ double block_sum(double v, double *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = lane < NT / 32 ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

__device__ __forceinline__ int tier_size(int l, int C) {
    const double rho = l == 0 ? 0.08 : (l == 1 ? 0.30 : 0.95);
    int k = (int)nearbyint(rho * C);  // round half to even
    k = k < 2 ? 2 : k;
    return k > C ? C : k;
}

// Eqs. 10-13 for one head pair of one sequence: rank its non-anchor chunks by q and
// sum the gains of the upgrades L -> M and M -> H.  Writes rank[c] (-1 for the
// anchors) and gains[2] = {gain_LM, gain_MH}.
__global__ void __launch_bounds__(kThreads)
selector_pair_kernel(const float *__restrict__ score, const float *__restrict__ g, const float *__restrict__ gamma,
                     const float *__restrict__ eta, int T_, int Nv, int C, int npow2, int32_t *__restrict__ rank_ws,
                     double *__restrict__ gains) {
    extern __shared__ unsigned long long keys[];  // [npow2]
    __shared__ float norm[2];
    __shared__ double L[2], G[2], rr[2], red[kThreads / 32], red2[kThreads / 32];
    const int p = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    pdl_wait();  // the intra step's scores
    pdl_trigger();
    const int h0 = 2 * p;
    const float *s0 = score + ((int64_t)b * Nv + h0) * C;
    const float *s1 = s0 + C;
    int32_t *rank = rank_ws + ((int64_t)b * kPairs + p) * C;

    // Eq. 11 for the two heads, each by half of the CTA (256 threads)
    const int half = tid >> 8, ht = tid & 255;
    const int h = h0 + half;
    const float *sh = half ? s1 : s0;
    double ss = 0.0;
    for (int c = ht; c < C; c += 256) ss += (double)sh[c] * (double)sh[c];
    // r_h: mean of 2^gamma over the last min(16, C) chunks
    const int c0 = C > 16 ? C - 16 : 0;
    double e2 = 0.0;
    if (ht < C - c0)  // gamma of chunk c0 + ht: given, or g at its last token (a partial last chunk ends at T - 1)
        e2 = exp2((double)(gamma ? gamma[((int64_t)b * Nv + h) * C + c0 + ht]
                                 : g[((int64_t)b * T_ + min((int64_t)(c0 + ht + 1) * kChunk, (int64_t)T_) - 1) * Nv + h]));
    // both half-sums at once: lanes reduce within the warp, warps of a half combine in shared memory
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        e2 += __shfl_xor_sync(0xffffffffu, e2, o);
    }
    if ((tid & 31) == 0) { red[tid >> 5] = ss; red2[tid >> 5] = e2; }
    __syncthreads();
    if (ht == 0) {
        double a = 0.0, r = 0.0;
        for (int w8 = 0; w8 < 8; ++w8) { a += red[8 * half + w8]; r += red2[8 * half + w8]; }
        norm[half] = sqrtf((float)a);
        rr[half] = C > c0 ? r / (C - c0) : 0.0;
    }
    __syncthreads();
    // L_h = sum_{j=1}^{C-2} r^j: thread ht sums the powers j in its segment
    {
        const double r = rr[half];
        const int n = C - 2, m = (n + 255) / 256;
        const int j0 = ht * m + 1, j1 = min(n, j0 + m - 1);
        double part = 0.0;
        if (j0 <= j1 && r > 0.0) {
            double pw = ipow(r, j0);
            for (int j = j0; j <= j1; ++j) { part += pw; pw *= r; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        __syncthreads();
        if ((tid & 31) == 0) red[tid >> 5] = part;
        __syncthreads();
        if (ht == 0) {
            double Lh = 0.0;
            for (int w8 = 0; w8 < 8; ++w8) Lh += red[8 * half + w8];
            double Gh = 1.0;
            if (eta) {
                double em = 0.0;
                for (int j = 0; j < Nv; ++j) em += (double)eta[(int64_t)b * Nv + j];
                em /= Nv;
                Gh = em > 0.0 ? sqrt((double)eta[(int64_t)b * Nv + h] / em) : 0.0;
            }
            L[half] = Lh;
            G[half] = Gh;
        }
    }
    __syncthreads();
    const int n_in = C > 2 ? C - 2 : 0;
    const float n0 = norm[0], n1 = norm[1];
    // Eq. 10: rank keys of the non-anchor chunks 1 .. C-2
    for (int i = tid; i < npow2; i += kThreads) {
        unsigned long long key = ~0ull;
        if (i < n_in) {
            const int c = i + 1;
            const float a0 = n0 > 0.f ? s0[c] / n0 : 0.f;
            const float a1 = n1 > 0.f ? s1[c] / n1 : 0.f;
            const float q = 0.5f * (a0 + a1);
            key = ((unsigned long long)(~__float_as_uint(q)) << 32) | (unsigned)c;
        }
        keys[i] = key;
    }
    __syncthreads();
    for (int size = 2; size <= npow2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < npow2; i += kThreads) {
                const int jx = i ^ stride;
                if (jx > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long x = keys[i], y = keys[jx];
                    if ((x > y) == up) { keys[i] = y; keys[jx] = x; }
                }
            }
            __syncthreads();
        }
    }
    // ranks, and the Eq. 12 gains of the upgrades L -> M (ranks [k_L-2, k_M-2)) and
    // M -> H (ranks [k_M-2, k_H-2))
    const double L0 = L[0], L1 = L[1], G0 = G[0], G1 = G[1];
    const int kL = tier_size(0, C) - 2, kM = tier_size(1, C) - 2, kH = tier_size(2, C) - 2;
    double wLM = 0.0, wMH = 0.0;
    for (int i = tid; i < n_in; i += kThreads) {
        const int c = (int)(keys[i] & 0xffffffffu);
        rank[c] = i;
        const double w = (double)s0[c] * L0 * G0 + (double)s1[c] * L1 * G1;
        if (i >= kL && i < kM) wLM += w;
        if (i >= kM && i < kH) wMH += w;
    }
    if (tid == 0 && C > 0) {
        rank[0] = -1;
        rank[C - 1] = -1;
    }
    const double tLM = block_sum<kThreads>(wLM, red);
    const double tMH = block_sum<kThreads>(wMH, red2);
    if (tid == 0) {
        gains[((int64_t)b * kPairs + p) * 2 + 0] = tLM;
        gains[((int64_t)b * kPairs + p) * 2 + 1] = tMH;
    }
}

// Eq. 14 for one sequence, then the mask of every pair: anchors plus its tier's
// best k - 2 chunks.  Thread p < 16 normalises pair p's gains and finds its place
// in the descending orders; candidate counts are scored one per thread.
__global__ void __launch_bounds__(256)
selector_tier_kernel(int C, const int32_t *__restrict__ rank_ws, const double *__restrict__ gains,
                     uint8_t *__restrict__ mask, int32_t *__restrict__ tier_out) {
    __shared__ double gLM[kPairs], gMH[kPairs], xM[kPairs], xH[kPairs], xs[kPairs], sep[kPairs];
    __shared__ int ids[kPairs], rest[kPairs], tier[kPairs], kk[3], nH_s, nr_s;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();  // the pair kernel's ranks and gains
    pdl_trigger();
    if (tid < kPairs) {
        gLM[tid] = gains[((int64_t)b * kPairs + tid) * 2];
        gMH[tid] = gains[((int64_t)b * kPairs + tid) * 2 + 1];
        ids[tid] = tid;
    }
    if (tid < 3) kk[tid] = tier_size(tid, C);
    __syncthreads();
    if (tid < 32) {  // means over the 16 pairs by a shuffle tree, then x = gain / mean
        double mLM = tid < kPairs ? gLM[tid] : 0.0, mMH = tid < kPairs ? gMH[tid] : 0.0;
#pragma unroll
        for (int o = 8; o; o >>= 1) {
            mLM += __shfl_xor_sync(0xffffffffu, mLM, o);
            mMH += __shfl_xor_sync(0xffffffffu, mMH, o);
        }
        mLM /= kPairs;
        mMH /= kPairs;
        if (tid < kPairs) {
            xM[tid] = mLM != 0.0 ? gLM[tid] / mLM : 0.0;
            xH[tid] = mMH != 0.0 ? gMH[tid] / mMH : 0.0;
        }
    }
    __syncthreads();
    // high tier: x_H sorted descending, B(x_H, k) for k = 1..4, the first maximum wins
    if (tid < kPairs) {
        const int pos = desc_position(xH, ids, kPairs, tid);
        xs[pos] = xH[tid];
        rest[pos] = tid;  // pair at each position of the x_H order
    }
    __syncthreads();
    if (tid < 4) sep[tid] = separation(xs, kPairs, tid + 1);
    __syncthreads();
    if (tid == 0) {
        int nH = 1;
        for (int k = 2; k <= 4; ++k)
            if (sep[k - 1] > sep[nH - 1]) nH = k;
        nH_s = nH;
        for (int p = 0; p < kPairs; ++p) tier[p] = 0;
        for (int i = 0; i < nH; ++i) tier[rest[i]] = 2;
        int nr = 0;
        for (int p = 0; p < kPairs; ++p)
            if (tier[p] != 2) ids[nr++] = p;  // the remaining pairs, in pair order
        nr_s = nr;
    }
    __syncthreads();
    // mid tier among the rest: x_M sorted descending, B over the table row of n_H
    const int nH = nH_s, nr = nr_s;
    const int lo = nH == 1 ? 11 : (nH == 2 ? 7 : (nH == 3 ? 3 : 0));
    const int hi = nH == 1 ? 13 : (nH == 2 ? 9 : (nH == 3 ? 5 : 0));
    if (tid < nr) {
        const int pos = desc_position(xM, ids, nr, tid);
        xs[pos] = xM[ids[tid]];
        rest[pos] = ids[tid];
    }
    __syncthreads();
    if (hi > 0 && tid <= hi - lo) sep[tid] = separation(xs, nr, lo + tid);
    __syncthreads();
    if (tid == 0) {
        int nM = 0;
        if (hi > 0) {
            nM = lo;
            for (int k = lo + 1; k <= hi; ++k)
                if (sep[k - lo] > sep[nM - lo]) nM = k;
        }
        for (int i = 0; i < nM; ++i) tier[rest[i]] = 1;
    }
    __syncthreads();
    if (tier_out && tid < kPairs) tier_out[(int64_t)b * kPairs + tid] = tier[tid];
    const int32_t *rk = rank_ws + (int64_t)b * kPairs * C;
    uint8_t *mb = mask + (int64_t)b * kPairs * C;
    for (int idx = tid; idx < kPairs * C; idx += blockDim.x) {
        const int p = idx / C;
        const int r = rk[idx];
        mb[idx] = (r < 0 || r < kk[tier[p]] - 2) ? 1 : 0;
    }
}

}  // namespace

size_t selector_workspace_bytes(int B, int C) {
    return (size_t)B * kPairs * 2 * sizeof(double) + (size_t)B * kPairs * C * sizeof(int32_t);
}

cudaError_t launch_selector(const Problem &pb, const float *score, const float *eta, uint8_t *mask,
                            int32_t *tier_out, void *ws, const float *gamma) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    int npow2 = 1;
    while (npow2 < (pb.C > 2 ? pb.C - 2 : 1)) npow2 <<= 1;
    const size_t smem = (size_t)npow2 * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(selector_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    double *gains = (double *)ws;                                    // [B,16,2]
    int32_t *rank = (int32_t *)(gains + (size_t)pb.B * kPairs * 2);  // [B,16,C]
    e = launch_kernel(pb.pdl, selector_pair_kernel, dim3(kPairs, pb.B), kThreads, smem, pb.stream, score, pb.g, gamma,
                      eta, pb.T, pb.Nv, pb.C, npow2, rank, gains);
    if (e != cudaSuccess) return e;
    return launch_kernel(pb.pdl_ok, selector_tier_kernel, pb.B, 256, 0, pb.stream, pb.C, (const int32_t *)rank,
                         (const double *)gains, mask, tier_out);
}

}  // namespace gdn
