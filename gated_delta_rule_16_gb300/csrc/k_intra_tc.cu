// k_intra_tc.cu -- intra-chunk step (SparseGDN Sec. 2.3, Eqs. 5-9) on tcgen05
// tensor cores, for bf16 storage.
//
// One CTA per (group of two chunks, head pair, sequence): 128 tokens, 256 threads,
// ~110 KB of shared memory and 256 TMEM columns, so two CTAs share an SM and one
// CTA's loads, barriers and MMA round trips overlap the other's work.  The pair's two
// value heads share the key head, so the K tile, the Gram product and the CTA's
// set-up serve both; the heads then run one after the other, and the second head's V
// tile loads while its M and solve proceed.
//   Gram  G = K K^T [128 x 128]        (A = B = the K tile, K-major, by TMA)
//   A_Delta[t,s] = beta_t G[t,s] 2^(g_t - g_s), s < t in the same chunk; M = I + A_Delta
//   C = M^-1 (exact) or the block-adjacent approximation (Eq. 7), fp32 over compact
//       16x16 blocks: C_ii = M_ii^-1 (8x8 forward substitutions and two 8x8 products on CUDA cores),
//       C_ij = -C_ii sum_{k=j}^{i-1} M_ik C_kj (the block-adjacent solver's two products
//       per block on the warps' tensor cores in three-pass tf32, nearly fp32 accuracy)
//   U = C diag(beta) V                  (A: C diag(beta) bf16, block-diagonal over the
//                                        two chunks, K-major; B: V [tok][dv] MN-major by TMA)
//   s = ||U[48:64,:]||_F (Tail-16 write score)
//   W = C diag(beta 2^g) K for the chunks that are events (Eq. 15): A = C-bar bf16,
//       block-diagonal, K-major, built in the V tile once the U product has read it;
//       B = the K tile read as MN-major (token rows, d columns: the same bytes as the
//       K-major Gram operand).  W is built only for event chunks and stored negated
//       (the scan accumulates -S^T W^T onto U^T).  W of (row i = b P + p, chunk c) lives
//       at slot i C + c, so this kernel needs only the caller's mask, not the compaction.
// Shared memory over the CTA's life:
//   [0, 32K)     K tile (Gram, then the W products)
//   [32K, 64K)   per head: V tile -> C-bar operand -> W staging
//   [64K, 106K)  per head: solver blocks (fp32) -> C diag(beta) operand (first 32K) -> U staging
// TMEM: the Gram at columns 0-127 for both heads; each head's U, then W, at 128-255.
// Each thread keeps its row's 32 coefficients of C in registers between the solve and
// the two operand builds, which is what lets the operands overwrite the solver blocks.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 256;  // 8 warps: 2 per TMEM lane quarter, 64 columns each
constexpr uint32_t kSlab = 16384;
constexpr uint32_t OFF_K = 0;            // K tile: 2 K-slabs [128 tok][64 d]
constexpr uint32_t OFF_V = 2 * kSlab;    // V tile of the head: 2 MN-stacks [128 tok][64 dv]
constexpr uint32_t OFF_A = 4 * kSlab;    // solver blocks, then C diag(beta) bf16: 2 K-slabs [128 t][64 s]
// Solver blocks: 16x16 fp32 with a row stride of 20 floats (16-byte rows; eight rows read
// at the same column quad fall in distinct banks), slots 16 floats apart beyond that so
// that neighbouring blocks start 16 banks apart (the two half-warps of the diagonal solve
// read two blocks at once).  Per chunk: the 4 diagonal blocks (M_ii, then C_ii in place),
// the 6 below-diagonal blocks of M and the 6 of C.
constexpr int BS = 20;
constexpr int kBlkFloats = kBlk * BS + 16;
constexpr int kSlots = 16;
constexpr uint32_t kSolveBytes = 2 * kSlots * kBlkFloats * 4;
constexpr uint32_t OFF_SMALL = OFF_A + kSolveBytes;  // beta, g, beta 2^g of the 128 tokens, both heads
constexpr uint32_t kIntraTcSmem = 1024 + OFF_SMALL + 3 * 2 * 128 * 4;
static_assert(kSolveBytes >= 2 * kSlab, "the U operand and staging reuse the solver blocks");
static_assert(kIntraTcSmem + 1024 <= 114 * 1024, "two CTAs per SM");
constexpr uint32_t TM_G = 0, TM_U = 128;  // W reuses the U columns

struct IntraParams {
    const float *beta, *g;
    const uint8_t *mask;    // [B,P,C] event mask, NULL: every chunk is an event
    int build_w;            // 0: no W here (it is built later from C-bar)
    __nv_bfloat16 *U, *W;
    __nv_bfloat16 *cbar;    // non-NULL: write the compact C-bar blocks [B,Nv,C,nblk,16,16] (bf16)
    float *score;
    int32_t *status;
    const int32_t *row_pair;  // non-NULL: blockIdx.y is CSR row row0 + y (pair row_pair[row0 + y])
    int row0;
    int P_, T_, Nv, C, nblk, exact, tail;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Solver block addresses inside the fp32 area F (chunk cc, block row ib, block column jb).
__device__ __forceinline__ int below(int ib, int jb) { return ib * (ib - 1) / 2 + jb; }
__device__ __forceinline__ float *blk_diag(float *F, int cc, int ib) { return F + (cc * kSlots + ib) * kBlkFloats; }
__device__ __forceinline__ float *blk_m(float *F, int cc, int ib, int jb) {
    return F + (cc * kSlots + 4 + below(ib, jb)) * kBlkFloats;
}
__device__ __forceinline__ float *blk_c(float *F, int cc, int ib, int jb) {
    return F + (cc * kSlots + 10 + below(ib, jb)) * kBlkFloats;
}
__device__ __forceinline__ float *blk_cc(float *F, int cc, int ib, int jb) {
    return ib == jb ? blk_diag(F, cc, ib) : blk_c(F, cc, ib, jb);
}
// Index of block (ib, jb) in the compact C-bar order (diagonal, sub-diagonal, far).
__device__ __forceinline__ int cbar_index(int ib, int jb) {
    return ib == jb ? ib : (jb + 1 == ib ? 3 + ib : (ib == 2 ? 7 : (jb == 1 ? 8 : 9)));
}

// Below-diagonal blocks of C, one warp per block: T = sum_{k=jb}^{ib-1} M_{ib,k} C_{k,jb}, then
// C_{ib,jb} = -C_{ib,ib} T (Eq. 7; the block-adjacent solver keeps ib = jb + 1 only), each a sum of
// 16x16x16 products on the warp's tensor cores (mma m16n8k8 in tf32, fp32 accumulation).
// Every factor is split into a tf32 head and a tf32 tail (x = hi + lo up to about 2^-22 |x|) and a
// product takes the three terms lo*hi, hi*lo, hi*hi (the dropped lo*lo is about 2^-22 of it), so it
// carries nearly fp32 accuracy.  Lane (g = lane / 4,
// q = lane % 4) holds A[g][q], A[g+8][q], A[g][q+4], A[g+8][q+4] of each 16x8 A slice, B[q][n], B[q+4][n]
// (n = g) of each 8x8 B slice and D[g][2q], D[g][2q+1], D[g+8][2q], D[g+8][2q+1] of each 16x8 result.
// T goes over M's block (only this warp reads it) between the two products.
__device__ __forceinline__ uint32_t tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D[16 x 16] += A[16 x 16] B[16 x 16], both read from solver blocks (row stride BS).
__device__ __forceinline__ void prod16_3xtf32(const float *A, const float *B, int lane, float (&d)[2][4]) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 8) {
        const float av[4] = {A[g * BS + kk + q], A[(g + 8) * BS + kk + q], A[g * BS + kk + q + 4],
                             A[(g + 8) * BS + kk + q + 4]};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ah[e] = tf32_hi(av[e]);
            al[e] = tf32_hi(av[e] - __uint_as_float(ah[e]));
        }
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
            const float b0 = B[(kk + q) * BS + nn * 8 + g], b1 = B[(kk + q + 4) * BS + nn * 8 + g];
            const uint32_t bh0 = tf32_hi(b0), bh1 = tf32_hi(b1);
            const uint32_t bl0 = tf32_hi(b0 - __uint_as_float(bh0)), bl1 = tf32_hi(b1 - __uint_as_float(bh1));
            mma_tf32(d[nn], al, bh0, bh1);
            mma_tf32(d[nn], ah, bl0, bl1);
            mma_tf32(d[nn], ah, bh0, bh1);
        }
    }
}
// The blocks at distance OFF below the diagonal of both chunks (warp w < 2 (4 - OFF): chunk
// w / (4 - OFF), block column jb = w % (4 - OFF), row ib = jb + OFF); every block closer to the
// diagonal is known.  T goes to C's block (only this warp reads it) and C replaces it there.
template <int OFF>
__device__ __forceinline__ void offdiag_level(float *F, int warp, int lane) {
    constexpr int NB = 4 - OFF;
    if (warp < 2 * NB) {
        const int cc = warp / NB, jb = warp % NB, ib = jb + OFF;
        const int g = lane >> 2, q = lane & 3;
        float d[2][4] = {};
#pragma unroll
        for (int kb = 0; kb < OFF; ++kb) prod16_3xtf32(blk_m(F, cc, ib, jb + kb), blk_cc(F, cc, jb + kb, jb), lane, d);
        float *Cb = blk_c(F, cc, ib, jb);
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
            *reinterpret_cast<float2 *>(Cb + g * BS + nn * 8 + 2 * q) = make_float2(d[nn][0], d[nn][1]);
            *reinterpret_cast<float2 *>(Cb + (g + 8) * BS + nn * 8 + 2 * q) = make_float2(d[nn][2], d[nn][3]);
        }
        __syncwarp();  // T complete
        float e[2][4] = {};
        prod16_3xtf32(blk_diag(F, cc, ib), Cb, lane, e);
        __syncwarp();  // every lane has read T
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
            *reinterpret_cast<float2 *>(Cb + g * BS + nn * 8 + 2 * q) = make_float2(-e[nn][0], -e[nn][1]);
            *reinterpret_cast<float2 *>(Cb + (g + 8) * BS + nn * 8 + 2 * q) = make_float2(-e[nn][2], -e[nn][3]);
        }
    }
}

// One row's 32 operand columns (this thread's half of its chunk) as bf16 into the
// chunk's slab, and zeros into the other chunk's slab (the tile is block-diagonal).
__device__ __forceinline__ void build_operand_row(uint8_t *tile, int row, int ct, int half, const float *creg,
                                                  const float *fcol) {
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) {
        const float4 f0 = ld4(fcol + k0), f1 = ld4(fcol + k0 + 4);
        const float w[8] = {creg[k0] * f0.x,     creg[k0 + 1] * f0.y, creg[k0 + 2] * f0.z, creg[k0 + 3] * f0.w,
                            creg[k0 + 4] * f1.x, creg[k0 + 5] * f1.y, creg[k0 + 6] * f1.z, creg[k0 + 7] * f1.w};
        st_sw128_8(tile + ct * kSlab, row, 32 * half + k0, w);
        st_sw128_8(tile + (1 - ct) * kSlab, row, 32 * half + k0, z);
    }
}

__global__ void __launch_bounds__(kThreads, 2)
intra_tc_kernel(const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
                const __grid_constant__ CUtensorMap tU, const __grid_constant__ CUtensorMap tW, IntraParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_ld, bar_v, bar_g, bar_u, bar_w, bar_drain;
    __shared__ int ev_s[2];
    __shared__ float ssum_w[kThreads / 32];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    float *F = reinterpret_cast<float *>(sm + OFF_A);
    float *bet2 = reinterpret_cast<float *>(sm + OFF_SMALL);  // [head][token]
    float *gg2 = bet2 + 256;
    float *bgs2 = gg2 + 256;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter; which 64 of 128 columns
    const int row = quarter * 32 + lane;             // token inside the group
    const int ct = row >> 6, tl = row & 63, ib = tl >> 4, rr = tl & 15;
    const int r = blockIdx.x;
    const int pr = a.row_pair ? a.row_pair[a.row0 + blockIdx.y] : 0;
    const int p = a.row_pair ? pr % a.P_ : (int)blockIdx.y, b = a.row_pair ? pr / a.P_ : (int)blockIdx.z;
    const int c0 = 2 * r;
    const int nch = c0 + 1 < a.C ? 2 : 1;
    const int t0 = c0 * kChunk;                        // first token of the group inside its sequence
    const int nvalid = min(2 * kChunk, a.T_ - t0);     // tokens of the group (a partial last chunk has fewer)
    const int64_t tok0 = (int64_t)b * a.T_ + t0;
    // Tail-W window of this thread's row: the last W valid rows of its chunk (rows past the
    // sequence's end need no exclusion: beta = 0 there makes their U rows exactly zero)
    const int nrow = min(kChunk, nvalid - kChunk * ct);
    const bool in_tail = tl >= nrow - a.tail;
    const bool exact = a.exact != 0;

    pdl_trigger();
    if (tid == 0) {  // barriers, then the tiles: the loads overlap the set-up below
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_u, 1);
        mbar_init(&bar_w, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        abort_s = 0;
        mbar_arrive_expect_tx(&bar_ld, 2 * kSlab);  // K: the Gram product starts once it lands
        tma_load_4d(sm + OFF_K, &tK, 0, p, t0, b, &bar_ld);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_K + kSlab, &tK, 64, p, t0, b, &bar_ld);
        mbar_arrive_expect_tx(&bar_v, 2 * kSlab);   // V of the first head: needed only by its U product
        tma_load_4d(sm + OFF_V, &tV, 0, 2 * p, t0, b, &bar_v);
        tma_load_4d(sm + OFF_V + kSlab, &tV, 64, 2 * p, t0, b, &bar_v);
    }
    if (tid >= kThreads - 2) {  // the W slot of each event chunk of the group, else -1
        const int cc = tid - (kThreads - 2);
        const int64_t slot = ((int64_t)b * a.P_ + p) * a.C + c0 + cc;
        ev_s[cc] = a.build_w && cc < nch && (!a.mask || a.mask[slot]) ? (int)slot : -1;
    }
    {   // beta and g of both heads, fetched while the tiles load; tokens past the sequence's
        // end: beta = 0 (no write, no correction) and a finite g
        const int t = tid & 127;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int64_t gi = (tok0 + min(t, nvalid - 1)) * a.Nv + 2 * p + hh;
            if (tid < 128) bet2[128 * hh + t] = t < nvalid ? a.beta[gi] : 0.f;
            else gg2[128 * hh + t] = a.g[gi];
        }
    }
    if (warp == 0) tmem_alloc<256>(&tmem_base);
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
    bgs2[tid] = bet2[tid] * ex2(gg2[tid]);
    __syncthreads();
    if (!abort_s && !mbar_wait(&bar_g, 0)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
    tc_fence_after();
    int v_loads = 1;  // V tiles requested (thread 0)
    for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * p + hh;
        const float *bet = bet2 + 128 * hh, *gg = gg2 + 128 * hh, *bgs = bgs2 + 128 * hh;
        tc_fence_after();
        // 1. M from the Gram block of the row's chunk: thread (row, half) covers blocks 2 half, 2 half + 1
        {
            float gv[32];
            tmem_ld32(tmem_addr(tbase, quarter * 32, TM_G + 64 * ct + 32 * half), gv);
            tmem_ld_wait();
            const float bt = bet[row], gt = gg[row];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int jb = 2 * half + h2;
                if (jb <= ib && (exact || jb + 1 >= ib)) {
                    float *dst = (jb == ib ? blk_diag(F, ct, ib) : blk_m(F, ct, ib, jb)) + rr * BS;
                    float v[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int s = 16 * jb + c;
                        v[c] = s < tl ? bt * gv[16 * h2 + c] * ex2(gt - gg[64 * ct + s]) : (s == tl ? 1.f : 0.f);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<float4 *>(dst + 4 * q4) =
                            make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        // 2. solve.  Diagonal 16x16 blocks, in place: warp w < 4 takes blocks 2w and 2w+1 (8 blocks:
        //    2 chunks x 4), lanes 16 (w' = lane / 16) apart.  Split into 8x8 sub-blocks,
        //    M_ii = [[A, 0], [B, D]], its inverse is [[A^-1, 0], [-D^-1 B A^-1, D^-1]]:
        //    (a) A^-1 and D^-1 by forward substitution, one lane per column of a sub-block (rows of the
        //        sub-block broadcast from shared memory): X[i][j] = -sum_{s<i} M[i][s] X[s][j];
        //    (b) the lower-left quarter as two 8x8 products, lane (row r, four columns).
        if (warp < 4) {
            float *Mb = blk_diag(F, (2 * warp + (lane >> 4)) >> 2, (2 * warp + (lane >> 4)) & 3);
            {   // (a)
                const int sub = (lane >> 3) & 1, j = lane & 7;
                float *Sb = Mb + sub * (8 * BS + 8);
                float x[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) x[i2] = i2 == j ? 1.f : 0.f;
#pragma unroll
                for (int i2 = 1; i2 < 8; ++i2) {
                    float mr[8];  // row i2 of the sub-block, 16-byte loads (broadcast across its 8 lanes)
#pragma unroll
                    for (int q4 = 0; q4 < (i2 + 3) / 4; ++q4) {
                        const float4 m4 = ld4(Sb + i2 * BS + 4 * q4);
                        mr[4 * q4] = m4.x; mr[4 * q4 + 1] = m4.y; mr[4 * q4 + 2] = m4.z; mr[4 * q4 + 3] = m4.w;
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < i2; ++s2) acc += mr[s2] * x[s2];
                    if (i2 > j) x[i2] = -acc;
                }
                __syncwarp();  // every lane has read its sub-block before the inverse replaces it
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) Sb[i2 * BS + j] = x[i2];
                __syncwarp();
            }
            {   // (b) T = B A^-1 over B, then -D^-1 T over T
                const int r = (lane >> 1) & 7, c4 = (lane & 1) * 4;
                float *Bq = Mb + 8 * BS;           // rows 8..15, columns 0..7
                const float *XA = Mb, *XD = Mb + 8 * BS + 8;
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                {
                    const float4 b0 = ld4(Bq + r * BS), b1 = ld4(Bq + r * BS + 4);
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 xa = ld4(XA + k * BS + c4);
                        t.x += bv[k] * xa.x; t.y += bv[k] * xa.y; t.z += bv[k] * xa.z; t.w += bv[k] * xa.w;
                    }
                }
                __syncwarp();  // every lane has read B
                *reinterpret_cast<float4 *>(Bq + r * BS + c4) = t;
                __syncwarp();  // T complete
                float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
                {
                    const float4 d0 = ld4(XD + r * BS), d1 = ld4(XD + r * BS + 4);
                    const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 tk = ld4(Bq + k * BS + c4);
                        l.x += dv[k] * tk.x; l.y += dv[k] * tk.y; l.z += dv[k] * tk.z; l.w += dv[k] * tk.w;
                    }
                }
                __syncwarp();  // every lane has read T
                *reinterpret_cast<float4 *>(Bq + r * BS + c4) = make_float4(-l.x, -l.y, -l.z, -l.w);
            }
        }
        __syncthreads();
        offdiag_level<1>(F, warp, lane);
        __syncthreads();
        if (exact) {
            offdiag_level<2>(F, warp, lane);
            __syncthreads();
            offdiag_level<3>(F, warp, lane);
            __syncthreads();
        }
        const bool any_event = ev_s[0] >= 0 || ev_s[1] >= 0;
        // 3. this thread's 32 coefficients of C (blocks the solver does not keep are zero)
        float creg[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int jb = 2 * half + h2;
            if (jb <= ib && (exact || jb + 1 >= ib)) {
                const float *src = blk_cc(F, ct, ib, jb) + rr * BS;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 x = ld4(src + 4 * q4);
                    creg[16 * h2 + 4 * q4] = x.x;
                    creg[16 * h2 + 4 * q4 + 1] = x.y;
                    creg[16 * h2 + 4 * q4 + 2] = x.z;
                    creg[16 * h2 + 4 * q4 + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c) creg[16 * h2 + c] = 0.f;
            }
        }
        __syncthreads();  // the operand below overwrites the solver blocks
        // 4. A = C diag(beta) for U; the compact C-bar blocks for a later W kernel (online selection)
        build_operand_row(sm + OFF_A, row, ct, half, creg, bet + 64 * ct + 32 * half);
        if (a.cbar && ct < nch) {  // C-bar = C diag(beta 2^g), bf16 as in the W operand
            const float *gcol = bgs + 64 * ct + 32 * half;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int jb = 2 * half + h2;
                if (jb <= ib && (exact || jb + 1 >= ib)) {  // one block row: 32 bytes, a whole sector
                    uint32_t w[8];
#pragma unroll
                    for (int q2 = 0; q2 < 8; ++q2)
                        w[q2] = pack_bf16x2(creg[16 * h2 + 2 * q2] * gcol[16 * h2 + 2 * q2],
                                            creg[16 * h2 + 2 * q2 + 1] * gcol[16 * h2 + 2 * q2 + 1]);
                    st_global_v8(a.cbar + (((int64_t)b * a.Nv + h) * a.C + c0 + ct) * a.nblk * 256 +
                                     cbar_index(ib, jb) * 256 + rr * 16,
                                 w);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // 5. U = (C diag(beta)) V
        const uint32_t id = idesc_bf16(128, 128, false, true);
        if (tid == 0 && !abort_s) {
            if (!mbar_wait(&bar_v, hh)) {
                abort_s = 1;
                atomicOr(a.status, kStatusTimeout);
            } else {
                tc_fence_after();
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_U, kmajor_desc(smem_addr(sm + OFF_A), ks, kSlab),
                             mnmajor_desc(smem_addr(sm + OFF_V), ks, kSlab), id, ks > 0);
                mma_commit(&bar_u);
            }
        }
        if (!abort_s && !mbar_wait(&bar_u, hh)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
        tc_fence_after();
        // 6. U rows staged over the A operand (read by now), the write score of the tail rows,
        //    and, for events, the C-bar operand built over the V tile (also read by now)
        {
            float sq = 0.f;
            uint8_t *ust = sm + OFF_A + half * kSlab;
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                float u[32];
                tmem_ld32(tmem_addr(tbase, quarter * 32, TM_U + 64 * half + 32 * s2), u);
                tmem_ld_wait();
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(ust, row, 32 * s2 + 8 * v8, &u[8 * v8]);
                if (in_tail) {
#pragma unroll
                    for (int q2 = 0; q2 < 32; ++q2) sq += u[q2] * u[q2];
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            if (lane == 0) ssum_w[warp] = sq;
        }
        if (any_event) build_operand_row(sm + OFF_V, row, ct, half, creg, bgs + 64 * ct + 32 * half);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // 7. U out (rows past the sequence's end are clipped); W = (C diag(beta 2^g)) K for events
        if (tid == 0 && !abort_s) {
            tma_store_4d(&tU, 0, t0, h, b, sm + OFF_A);
            tma_store_4d(&tU, 64, t0, h, b, sm + OFF_A + kSlab);
            bulk_commit();
            if (any_event) {
                tc_fence_after();
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_U, kmajor_desc(smem_addr(sm + OFF_V), ks, kSlab),
                             mnmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id, ks > 0);
                mma_commit(&bar_w);
            }
        }
        if (tid < nch && a.score) {  // the chunk's four warps, summed in a fixed order
            const int w0 = 2 * tid;
            const float s = ssum_w[w0] + ssum_w[w0 + 1] + ssum_w[w0 + 4] + ssum_w[w0 + 5];
            a.score[((int64_t)b * a.Nv + h) * a.C + c0 + tid] = sqrtf(s);
        }
        if (any_event) {
            if (!abort_s && !mbar_wait(&bar_w, hh)) { abort_s = 1; atomicOr(a.status, kStatusTimeout); }
            tc_fence_after();
            if (ev_s[ct] >= 0) {  // warp-uniform: W rows staged over the C-bar operand (read by now)
                uint8_t *wst = sm + OFF_V + half * kSlab;
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                    float w[32];
                    tmem_ld32(tmem_addr(tbase, quarter * 32, TM_U + 64 * half + 32 * s2), w);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) w[q] = -w[q];  // the workspace holds -W
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(wst, row, 32 * s2 + 8 * v8, &w[8 * v8]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0 && !abort_s) {
                for (int cc = 0; cc < nch; ++cc) {
                    const int ev = ev_s[cc];
                    if (ev < 0) continue;
                    const int wrow = (ev * 2 + hh) * kChunk;
                    tma_store_3d(&tW, 0, wrow, 0, sm + OFF_V + cc * 8192);
                    tma_store_3d(&tW, 64, wrow, 0, sm + OFF_V + kSlab + cc * 8192);
                }
                bulk_commit();
            }
        }
        if (tid == 0) {
            bulk_wait_read();  // the stores have read their shared-memory sources: V and solver areas free
            if (hh == 0 && !abort_s) {  // the second head's V tile, over the first head's last reader
                mbar_arrive_expect_tx(&bar_v, 2 * kSlab);
                tma_load_4d(sm + OFF_V, &tV, 0, h + 1, t0, b, &bar_v);
                tma_load_4d(sm + OFF_V + kSlab, &tV, 64, h + 1, t0, b, &bar_v);
                v_loads = 2;
            }
        }
        __syncthreads();
    }  // heads
    if (abort_s && tid == 0) {
        mbar_wait(&bar_ld, 0);
        mbar_wait(&bar_v, (v_loads - 1) & 1);
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    pdl_wait();  // also on an early exit: this grid's completion implies its predecessors'
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tbase);
}

}  // namespace

cudaError_t launch_intra_tc(const Problem &pb, const Workspace &ws, bool write_cbar) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tK, tV, tU, tW;
    const uint64_t wrows = (uint64_t)ws.ev_cap * 2 * kChunk;
    if (!make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 128) ||
        !make_tmap_tokens(&tV, pb.v, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_headmajor(&tU, ws.U, pb.Nv, pb.T, pb.B, 64, 128) ||
        !make_tmap_bf16_3d(&tW, ws.W, kDim, wrows, 1, kDim * 2, wrows * kDim * 2, 64, 64, 1))
        return cudaErrorInvalidValue;
    IntraParams a;
    // the masked full scan reads W of every chunk: build it for all of them
    a.beta = pb.beta; a.g = pb.g; a.mask = pb.scan_full ? nullptr : pb.mask; a.build_w = !write_cbar;
    a.cbar = write_cbar ? reinterpret_cast<__nv_bfloat16 *>(ws.cbar) : nullptr;
    a.U = (__nv_bfloat16 *)ws.U; a.W = (__nv_bfloat16 *)ws.W; a.score = pb.score;
    a.status = ws.counts + 2;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.nblk = pb.nblk;
    a.exact = pb.solver == GDN_SOLVER_EXACT;
    a.tail = pb.tail;
    a.row_pair = pb.nrows > 0 ? pb.row_pair : nullptr;
    a.row0 = pb.row0;
    cudaFuncSetAttribute(intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraTcSmem);
    const dim3 grid = pb.nrows > 0 ? dim3(pb.G, pb.nrows, 1) : dim3(pb.G, pb.P, pb.B);
    return launch_kernel(pb.pdl, intra_tc_kernel, grid, kThreads, kIntraTcSmem, pb.stream, tK, tV, tU, tW, a);
}

}  // namespace gdn
