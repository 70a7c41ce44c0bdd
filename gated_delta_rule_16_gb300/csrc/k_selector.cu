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
// scores are norms).  The gains are summed by one thread in rank order, so every
// decision is taken from the same fp32 q values and the same fp64 sums as the
// sequential definition and the masks are reproducible bit for bit.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;
constexpr int kPairs = 16;

__device__ double separation(const double *xs, int n, int k) {
    double top = 0.0, rest = 0.0;
    for (int i = 0; i < k; ++i) top += xs[i];
    for (int i = k; i < n; ++i) rest += xs[i];
    top /= k;
    rest = n > k ? rest / (n - k) : 0.0;
    return (double)k * (n - k) / n * (top - rest) * (top - rest);
}

// pair ids by x descending, ties to the lower id (insertion sort, n <= 16)
__device__ void order_pairs(const double *x, int *ids, int n) {
    for (int i = 1; i < n; ++i) {
        const int v = ids[i];
        int j = i - 1;
        while (j >= 0 && (x[ids[j]] < x[v] || (x[ids[j]] == x[v] && ids[j] > v))) {
            ids[j + 1] = ids[j];
            --j;
        }
        ids[j + 1] = v;
    }
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
selector_pair_kernel(const float *__restrict__ score, const float *__restrict__ g, const float *__restrict__ eta,
                     int T_, int Nv, int C, int npow2, int32_t *__restrict__ rank_ws, double *__restrict__ wbuf,
                     double *__restrict__ gains) {
    extern __shared__ unsigned long long keys[];  // [npow2]
    __shared__ float norm[2];
    __shared__ double L[2], G[2];
    const int p = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int h0 = 2 * p;
    const float *s0 = score + ((int64_t)b * Nv + h0) * C;
    const float *s1 = s0 + C;
    int32_t *rank = rank_ws + ((int64_t)b * kPairs + p) * C;
    double *w = wbuf + ((int64_t)b * kPairs + p) * C;

    // Eq. 11 for the two heads: thread j handles head h0 + j.  Every sum runs in index
    // order and every product is rounded on its own (no fused multiply-add), so the
    // fp64 values are those of the sequential definition.
    if (tid < 2) {
        const int h = h0 + tid;
        const float *sh = tid ? s1 : s0;
        double ss = 0.0;
        for (int c = 0; c < C; ++c) ss = __dadd_rn(ss, __dmul_rn((double)sh[c], (double)sh[c]));
        norm[tid] = sqrtf((float)ss);
        const int c0 = C > 16 ? C - 16 : 0;
        double r = 0.0;
        for (int c = c0; c < C; ++c)
            r = __dadd_rn(r, exp2((double)g[((int64_t)b * T_ + (int64_t)c * kChunk + kChunk - 1) * Nv + h]));
        r = C > c0 ? r / (C - c0) : 0.0;
        double Lh = 0.0, pw = 1.0;
        for (int j = 1; j <= C - 2; ++j) {
            pw = __dmul_rn(pw, r);
            Lh = __dadd_rn(Lh, pw);
        }
        double Gh = 1.0;
        if (eta) {
            double m = 0.0;
            for (int j = 0; j < Nv; ++j) m = __dadd_rn(m, (double)eta[(int64_t)b * Nv + j]);
            m /= Nv;
            Gh = m > 0.0 ? sqrt((double)eta[(int64_t)b * Nv + h] / m) : 0.0;
        }
        L[tid] = Lh;
        G[tid] = Gh;
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
    // ranks, and the Eq. 12 summands in rank order
    const double L0 = L[0], L1 = L[1], G0 = G[0], G1 = G[1];
    for (int i = tid; i < n_in; i += kThreads) {
        const int c = (int)(keys[i] & 0xffffffffu);
        rank[c] = i;
        w[i] = __dadd_rn(__dmul_rn(__dmul_rn((double)s0[c], L0), G0), __dmul_rn(__dmul_rn((double)s1[c], L1), G1));
    }
    if (tid == 0 && C > 0) {
        rank[0] = -1;
        rank[C - 1] = -1;
    }
    __syncthreads();
    // Eq. 12 in rank order: C_M \ C_L and C_H \ C_M (two threads, sequential sums)
    if (tid < 2) {
        const int lo = tier_size(tid, C) - 2, hi = tier_size(tid + 1, C) - 2;
        double t = 0.0;
        for (int i = lo; i < hi; ++i) t = __dadd_rn(t, w[i]);
        gains[((int64_t)b * kPairs + p) * 2 + tid] = t;
    }
}

// Eq. 14 for one sequence, then the mask of every pair: anchors plus its tier's
// best k - 2 chunks.
__global__ void __launch_bounds__(256)
selector_tier_kernel(int C, const int32_t *__restrict__ rank_ws, const double *__restrict__ gains,
                     uint8_t *__restrict__ mask, int32_t *__restrict__ tier_out) {
    __shared__ double xM[kPairs], xH[kPairs], xs[kPairs];
    __shared__ int ids[kPairs], rest[kPairs], tier[kPairs], kk[3];
    const int b = blockIdx.x, tid = threadIdx.x;
    if (tid == 0) {
        for (int l = 0; l < 3; ++l) kk[l] = tier_size(l, C);
        const double *gb = gains + (int64_t)b * kPairs * 2;
        double mLM = 0.0, mMH = 0.0;
        for (int p = 0; p < kPairs; ++p) { mLM += gb[2 * p]; mMH += gb[2 * p + 1]; }
        mLM /= kPairs;
        mMH /= kPairs;
        for (int p = 0; p < kPairs; ++p) {
            xM[p] = mLM != 0.0 ? gb[2 * p] / mLM : 0.0;
            xH[p] = mMH != 0.0 ? gb[2 * p + 1] / mMH : 0.0;
            ids[p] = p;
            tier[p] = 0;
        }
        order_pairs(xH, ids, kPairs);
        for (int i = 0; i < kPairs; ++i) xs[i] = xH[ids[i]];
        int nH = 1;
        double best = separation(xs, kPairs, 1);
        for (int k = 2; k <= 4; ++k) {
            const double v = separation(xs, kPairs, k);
            if (v > best) { best = v; nH = k; }
        }
        for (int i = 0; i < nH; ++i) tier[ids[i]] = 2;
        int nr = 0;
        for (int p = 0; p < kPairs; ++p)
            if (tier[p] != 2) rest[nr++] = p;
        order_pairs(xM, rest, nr);
        for (int i = 0; i < nr; ++i) xs[i] = xM[rest[i]];
        // admissible counts of mid-tier pairs for each high-tier count
        const int lo = nH == 1 ? 11 : (nH == 2 ? 7 : (nH == 3 ? 3 : 0));
        const int hi = nH == 1 ? 13 : (nH == 2 ? 9 : (nH == 3 ? 5 : 0));
        int nM = 0;
        if (hi > 0) {
            nM = lo;
            best = separation(xs, nr, lo);
            for (int k = lo + 1; k <= hi; ++k) {
                const double v = separation(xs, nr, k);
                if (v > best) { best = v; nM = k; }
            }
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
    return (size_t)B * kPairs * C * (sizeof(int32_t) + sizeof(double)) + (size_t)B * kPairs * 2 * sizeof(double);
}

cudaError_t launch_selector(const Problem &pb, const float *score, const float *eta, uint8_t *mask,
                            int32_t *tier_out, void *ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    int npow2 = 1;
    while (npow2 < (pb.C > 2 ? pb.C - 2 : 1)) npow2 <<= 1;
    const size_t smem = (size_t)npow2 * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(selector_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const size_t n = (size_t)pb.B * kPairs * pb.C;
    double *wbuf = (double *)ws;                  // [B,16,C] fp64, rank order
    double *gains = wbuf + n;                     // [B,16,2]
    int32_t *rank = (int32_t *)(gains + (size_t)pb.B * kPairs * 2);  // [B,16,C]
    selector_pair_kernel<<<dim3(kPairs, pb.B), kThreads, smem, pb.stream>>>(score, pb.g, eta, pb.T, pb.Nv, pb.C,
                                                                            npow2, rank, wbuf, gains);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    selector_tier_kernel<<<pb.B, 256, 0, pb.stream>>>(pb.C, rank, gains, mask, tier_out);
    return cudaGetLastError();
}

}  // namespace gdn
