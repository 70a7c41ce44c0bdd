// tc_unit.cu -- GPU unit test of the tcgen05 / TMA / TMEM building blocks in
// gated_delta_rule_16_gb300/csrc/tc.cuh: one 128 x N x 128 bf16 GEMM per launch,
// A K-major (TMA-loaded, or written by threads with the 128-byte swizzle),
// B K-major or MN-major (TMA-loaded), fp32 result read back from TMEM.
#include "../../gated_delta_rule_16_gb300/csrc/tc.cuh"
#include "../../gated_delta_rule_16_gb300/csrc/tmap.cuh"

using namespace gdn::tc;

namespace {

constexpr int kSmem = 1024 + 32768 + 65536;

__global__ void __launch_bounds__(128)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
               const float *__restrict__ Af32, int a_manual, int b_mn, int N, float *__restrict__ D,
               int *__restrict__ err) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;          // two K-slabs of [128 rows][128 B]
    uint8_t *sB = sm + 32768;  // K-major: two slabs of [N rows][128 B]; MN-major: N/64 stacks of [128 rows][128 B]
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int ok_s;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        ok_s = 1;
    }
    if (warp == 0) tmem_alloc<256>(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t b_bytes = (uint32_t)N * 256u;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, (a_manual ? 0u : 32768u) + b_bytes);
        if (!a_manual) {
            tma_load_3d(sA, &tA, 0, 0, 0, &bar_tma);
            tma_load_3d(sA + 16384, &tA, 64, 0, 0, &bar_tma);
        }
        if (b_mn) {
            for (int s = 0; s < N / 64; ++s) tma_load_3d(sB + s * 16384, &tB, 64 * s, 0, 0, &bar_tma);
        } else {
            tma_load_3d(sB, &tB, 0, 0, 0, &bar_tma);
            tma_load_3d(sB + N * 128, &tB, 64, 0, 0, &bar_tma);
        }
    }
    if (a_manual) {
        for (int k0 = 0; k0 < 128; k0 += 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = Af32[tid * 128 + k0 + j];
            st_sw128_8(sA + (k0 >> 6) * 16384, tid, k0 & 63, v);
        }
        fence_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        if (mbar_wait(&bar_tma, 0)) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, N, false, b_mn != 0);
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t ad = kmajor_desc(smem_addr(sA), ks, 16384);
                const uint64_t bd = b_mn ? mnmajor_desc(smem_addr(sB), ks, 16384)
                                         : kmajor_desc(smem_addr(sB), ks, (uint32_t)N * 128u);
                mma_bf16(tbase, ad, bd, idesc, ks > 0);
            }
            mma_commit(&bar_mma);
        } else {
            ok_s = 0;
            atomicExch(err, 1);
        }
    }
    __syncthreads();
    if (ok_s) {
        if (!mbar_wait(&bar_mma, 0)) {
            atomicExch(err, 2);
        } else {
            tc_fence_after();
            const int row = warp * 32 + (tid & 31);
            for (int c0 = 0; c0 < N; c0 += 32) {
                float v[32];
                tmem_ld32(tmem_addr(tbase, warp * 32, c0), v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) D[row * N + c0 + j] = v[j];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tbase);
}

}  // namespace

// A: bf16 [128][128] row-major (and the same values in fp32 for the thread-written path);
// B: b_mn ? bf16 [128][N] (K rows, N contiguous) : bf16 [N][128] (N rows, K contiguous).
extern "C" int tc_gemm(const void *A, const float *Af32, const void *B, int b_mn, int a_manual, int N, float *D,
                       int *err) {
    if (N != 64 && N != 128 && N != 256) return -1;
    CUtensorMap tA, tB;
    if (!gdn::make_tmap_bf16_3d(&tA, A, 128, 128, 1, 256, 128 * 256, 64, 128, 1)) return -2;
    bool okb = b_mn ? gdn::make_tmap_bf16_3d(&tB, B, N, 128, 1, (uint64_t)N * 2, (uint64_t)N * 256, 64, 128, 1)
                    : gdn::make_tmap_bf16_3d(&tB, B, 128, N, 1, 256, (uint64_t)N * 256, 64, N, 1);
    if (!okb) return -3;
    cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    tc_gemm_kernel<<<1, 128, kSmem>>>(tA, tB, Af32, a_manual, b_mn, N, D, err);
    if (cudaGetLastError() != cudaSuccess) return -4;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}
