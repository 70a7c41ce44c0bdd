// k_wbuild_tc.cu -- deferred W on tcgen05 tensor cores (SparseGDN Sec. 2.5, Eq. 15),
// for the prefill that selects its events online.
//
// The intra step stores, for every chunk and value head, the compact blocks of
// C-bar = C diag(beta 2^g) rounded to bf16 (the same values its own W operand
// would hold).  Once the events are known, this kernel builds W_e = C-bar_e K_e
// for every selected event e and both value heads of its pair.  One CTA takes
// two events per iteration, so that M = 128:
//   A_h = block-diag(C-bar_{e0,h}, C-bar_{e1,h})   [128 rows x 128 tokens] bf16, K-major,
//         assembled in shared memory from the compact blocks
//   B   = the two events' K tiles                  [128 tokens x 128 d] bf16, MN-major, by TMA
//   D_h = A_h B                                     fp32 in TMEM, columns 128 h .. 128 h + 127
// and writes -D_h rounded to bf16 at W rows (2 (i C + c) + h) * 64 by TMA, i the event's
// row and c its chunk (the workspace holds -W, which the scan's U' product accumulates
// onto U).  The event count is
// read on the device; the grid strides over event pairs.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 256;             // 8 warps: TMEM lane quarter w % 4, d half w / 4
constexpr uint32_t kSlab = 16384;
constexpr uint32_t OFF_K = 0;             // K tiles: 2 MN-stacks [128 tok][64 d]
constexpr uint32_t OFF_A = 2 * kSlab;     // A_h: 2 K-slabs [128 rows][64 tok] per head; W staging afterwards
constexpr uint32_t kWbuildSmem = 1024 + OFF_A + 4 * kSlab;
constexpr int kMaxGrid = 2048;

struct WbuildParams {
    const __nv_bfloat16 *cbar;   // [B, Nv, C, nblk, 16, 16]
    const int32_t *counts, *row_pair, *row_ptr, *ev_chunk;
    int32_t *status;
    int64_t ev_cap;
    int R, P_, T_, Nv, C, nblk;
};

__device__ __forceinline__ int find_row(const int32_t *row_ptr, int R, int e) {
    int lo = 0, hi = R - 1;  // largest j with row_ptr[j] <= e (rows may be empty)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (row_ptr[mid] <= e) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// compact index of block (ib, jb) of a 64x64 chunk matrix, or -1 if the solver drops it
__device__ __forceinline__ int blk_index(int ib, int jb, int nblk) {
    int k = -1;
    if (ib == jb) k = ib;
    else if (ib - jb == 1) k = 4 + jb;
    else if (ib == 2 && jb == 0) k = 7;
    else if (ib == 3 && jb == 1) k = 8;
    else if (ib == 3 && jb == 0) k = 9;
    return k < nblk ? k : -1;
}

__global__ void __launch_bounds__(kThreads, 2)
wbuild_tc_kernel(const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tW, WbuildParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_ld, bar_mma, bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int ev_b[2], ev_p[2], ev_c[2], ev_i[2], abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();  // C-bar and the event lists of the kernels before
    pdl_trigger();
    const int64_t E = min((int64_t)a.counts[0], a.ev_cap);
    const int64_t npairs = (E + 1) / 2;
    if (blockIdx.x >= npairs) return;

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 0) tmem_alloc<256>(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    uint32_t it = 0;
    for (int64_t pi = blockIdx.x; pi < npairs && !abort_s; pi += gridDim.x, ++it) {
        if (tid < 2) {
            const int64_t e = 2 * pi + tid;
            if (e < E) {
                const int j = find_row(a.row_ptr, a.R, (int)e);
                const int i = a.row_pair[j];
                ev_b[tid] = i / a.P_;
                ev_p[tid] = i % a.P_;
                ev_i[tid] = i;
                ev_c[tid] = a.ev_chunk[e];
            } else {
                ev_b[tid] = -1;
            }
        }
        if (tid == 0) bulk_wait_read();  // the previous W stores have left the staging area
        __syncthreads();
        const bool two = ev_b[1] >= 0;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_ld, (two ? 2 : 1) * 2 * 8192);
            for (int j = 0; j < (two ? 2 : 1); ++j) {
                const int t0 = ev_c[j] * kChunk;  // rows past the sequence's end read zeros
                tma_load_4d(sm + OFF_K + j * 8192, &tK, 0, ev_p[j], t0, ev_b[j], &bar_ld);
                tma_load_4d(sm + OFF_K + kSlab + j * 8192, &tK, 64, ev_p[j], t0, ev_b[j], &bar_ld);
            }
        }
        if (!two) {  // the absent event's token rows meet zero coefficients: make them finite zeros
            for (int idx = tid; idx < 2 * 512; idx += kThreads) {
                const int s = idx >> 9, c16 = idx & 511;
                *reinterpret_cast<uint4 *>(sm + OFF_K + s * kSlab + 8192 + c16 * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        // A_h: thread (row, slab); slab j holds event j's coefficients, the other slab zeros
        {
            const int row = tid >> 1, sl = tid & 1, j = row >> 6, t = row & 63;
            const int ib = t >> 4, rr = t & 15;
            const bool own = sl == j && ev_b[j] >= 0;
            for (int hh = 0; hh < 2; ++hh) {
                uint8_t *slab = sm + OFF_A + hh * 2 * kSlab + sl * kSlab;
                const __nv_bfloat16 *cb = nullptr;
                if (own)
                    cb = a.cbar + (((int64_t)ev_b[j] * a.Nv + 2 * ev_p[j] + hh) * a.C + ev_c[j]) * a.nblk * 256 +
                         rr * 16;
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
                    const int k = own ? blk_index(ib, jb, a.nblk) : -1;
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                    if (k >= 0) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(cb + k * 256);
                        lo = src[0];
                        hi = src[1];
                    }
                    *reinterpret_cast<uint4 *>(slab + sw128_offset(row, 16 * jb)) = lo;
                    *reinterpret_cast<uint4 *>(slab + sw128_offset(row, 16 * jb + 8)) = hi;
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            if (!mbar_wait(&bar_ld, it & 1)) {
                abort_s = 1;
                atomicOr(a.status, kStatusTimeout);
            } else {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 128, false, true);
                for (int hh = 0; hh < 2; ++hh)
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tbase + 128 * hh, kmajor_desc(smem_addr(sm + OFF_A + hh * 2 * kSlab), ks, kSlab),
                                 mnmajor_desc(smem_addr(sm + OFF_K), ks, kSlab), id, ks > 0);
                mma_commit(&bar_mma);
            }
        }
        __syncthreads();
        if (abort_s) break;
        if (!mbar_wait(&bar_mma, it & 1)) {
            atomicOr(a.status, kStatusTimeout);
            abort_s = 1;
        }
        tc_fence_after();
        __syncthreads();
        if (abort_s) break;
        {   // epilogue: rows 32 (w % 4) + lane, d half w / 4, both heads, staged over the A tiles
            const int quarter = warp & 3, dh = warp >> 2, row = quarter * 32 + lane;
            for (int hh = 0; hh < 2; ++hh) {
                uint8_t *stage = sm + OFF_A + hh * 2 * kSlab + dh * kSlab;
#pragma unroll
                for (int c32 = 0; c32 < 2; ++c32) {
                    float w[32];
                    tmem_ld32(tmem_addr(tbase, quarter * 32, 128 * hh + 64 * dh + 32 * c32), w);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) w[q] = -w[q];  // stored negated (see the header)
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) st_sw128_8(stage, row, 32 * c32 + 8 * v8, &w[8 * v8]);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            for (int j = 0; j < (two ? 2 : 1); ++j) {
                const int64_t slot = (int64_t)ev_i[j] * a.C + ev_c[j];  // W of (row i, chunk c)
                for (int hh = 0; hh < 2; ++hh) {
                    const int wrow = (int)((slot * 2 + hh) * kChunk);
                    uint8_t *stage = sm + OFF_A + hh * 2 * kSlab + j * 8192;
                    tma_store_3d(&tW, 0, wrow, 0, stage);
                    tma_store_3d(&tW, 64, wrow, 0, stage + kSlab);
                }
            }
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_read();
    if (abort_s && tid == 0) {  // let copies and MMAs in flight finish before the memory goes away
        mbar_wait(&bar_ld, (it & 1));
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tbase);
}

}  // namespace

cudaError_t launch_wbuild_tc(const Problem &pb, const Workspace &ws) {
    if (pb.B == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tK, tW;
    const uint64_t wrows = (uint64_t)ws.ev_cap * 2 * kChunk;
    if (!make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 64) ||
        !make_tmap_bf16_3d(&tW, ws.W, kDim, wrows, 1, kDim * 2, wrows * kDim * 2, 64, 64, 1))
        return cudaErrorInvalidValue;
    WbuildParams a;
    a.cbar = reinterpret_cast<const __nv_bfloat16 *>(ws.cbar);
    a.counts = ws.counts; a.row_pair = ws.row_pair; a.row_ptr = ws.row_ptr; a.ev_chunk = ws.ev_chunk;
    a.status = ws.counts + 2;
    a.ev_cap = ws.ev_cap;
    a.R = pb.R; a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.nblk = pb.nblk;
    const int64_t pairs = (ws.ev_cap + 1) / 2;
    const int grid = (int)(pairs < kMaxGrid ? pairs : kMaxGrid);
    cudaFuncSetAttribute(wbuild_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWbuildSmem);
    return launch_kernel(pb.pdl, wbuild_tc_kernel, grid, kThreads, kWbuildSmem, pb.stream, tK, tW, a);
}

}  // namespace gdn
