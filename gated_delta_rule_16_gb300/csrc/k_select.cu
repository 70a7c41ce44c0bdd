// k_select.cu -- event compaction: [B,P,C] mask -> CSR event lists
// (SparseGDN Sec. 2.5, Eq. 16: rows per head pair, events in time order,
// per-group predecessor event, device-resident event count).
//
// One CTA of 1024 threads does the whole batch: the mask is tiny (B*P*C bytes,
// 8 KiB at T = 32K) and the work is integer bookkeeping, so a single CTA with
// warp ballots and block scans keeps it to a few microseconds and bit-exact.
//
// Row order: event count descending, ties by physical row id ascending.
// Snapshot rule: event e (chunk c, next event of its row at chunk cn, or none)
// is some group's predecessor iff an even chunk index 2r with c < 2r <= cn
// exists and 2r <= 2(G-1); such events are numbered densely in event order.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int warp_incl_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Exclusive scan of a[0..n) into out[0..n] (out[n] = total), in shared memory.
__device__ void block_exclusive_scan(const int *a, int *out, int n, int *warp_tot) {
    int carry = 0;
    for (int base = 0; base < n; base += kThreads) {
        int i = base + threadIdx.x;
        int x = i < n ? a[i] : 0;
        int incl = warp_incl_scan(x);
        int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
            int ti = warp_incl_scan(t);
            warp_tot[lane] = ti - t;  // exclusive warp offsets
            if (lane == 31) warp_tot[32] = ti;
        }
        __syncthreads();
        if (i < n) out[i] = carry + warp_tot[warp] + incl - x;
        carry += warp_tot[32];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[n] = carry;
    __syncthreads();
}

__device__ __forceinline__ bool is_set(const uint8_t *mask, int64_t row, int C, int c) {
    return mask == nullptr ? true : mask[row * C + c] != 0;
}

__global__ void __launch_bounds__(kThreads)
select_kernel(const uint8_t *__restrict__ mask, int R, int C, int G,
              int32_t *__restrict__ row_pair, int32_t *__restrict__ row_ptr,
              int32_t *__restrict__ ev_chunk, int32_t *__restrict__ grp_pred,
              int32_t *__restrict__ snap_slot, int32_t *__restrict__ counts,
              int64_t ev_cap, int64_t snap_cap) {
    extern __shared__ int sm[];
    int *cnt = sm;               // [R]   events per physical row
    int *order = cnt + R;        // [R]   physical id of sorted row j
    int *sorted_cnt = order + R; // [R]
    int *ptr = sorted_cnt + R;   // [R+1] row offsets
    int *refc = ptr + R + 1;     // [R]   referenced events per sorted row
    int *refb = refc + R;        // [R+1] snapshot base per sorted row
    __shared__ int warp_tot[33];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // 1. events per row
    for (int i = warp; i < R; i += kWarps) {
        int n = 0;
        for (int c = lane; c < C; c += 32) n += is_set(mask, i, C, c);
#pragma unroll
        for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        if (lane == 0) cnt[i] = n;
    }
    __syncthreads();
    // 2. rank rows: count descending, id ascending (a total order: ranks are a permutation)
    for (int i = threadIdx.x; i < R; i += kThreads) {
        int ci = cnt[i], rank = 0;
        for (int j = 0; j < R; ++j) {
            int cj = cnt[j];
            rank += (cj > ci) || (cj == ci && j < i);
        }
        order[rank] = i;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < R; j += kThreads) sorted_cnt[j] = cnt[order[j]];
    __syncthreads();
    // 3. row offsets
    block_exclusive_scan(sorted_cnt, ptr, R, warp_tot);
    const int64_t E = ptr[R];
    // 4. per row: event chunks, predecessor of each group, referenced-event count
    for (int j = warp; j < R; j += kWarps) {
        const int i = order[j];
        const int base = ptr[j];
        int run = 0;  // events of this row with chunk < current word start
        for (int w0 = 0; w0 < C; w0 += 32) {
            const int c = w0 + lane;
            const bool s = c < C && is_set(mask, i, C, c);
            const unsigned bits = __ballot_sync(0xffffffffu, s);
            const int before = __popc(bits & ((1u << lane) - 1u));
            if (s && (int64_t)base + run + before < ev_cap) ev_chunk[base + run + before] = c;
            // groups r with 2r in [w0, w0+32): lane l < 16 handles 2r = w0 + 2l
            if (lane < 16) {
                const int r = (w0 >> 1) + lane;
                if (r < G) {
                    const int n_before = run + __popc(bits & ((1u << (2 * lane)) - 1u));
                    grp_pred[(int64_t)i * G + r] = n_before > 0 ? base + n_before - 1 : -1;
                }
            }
            run += __popc(bits);
        }
        // referenced events: need the next event's chunk, re-read from the mask
        int nref = 0;
        for (int w0 = 0; w0 < C; w0 += 32) {
            const int c = w0 + lane;
            const bool s = c < C && is_set(mask, i, C, c);
            const unsigned bits = __ballot_sync(0xffffffffu, s);
            bool ref = false;
            if (s) {
                const int m = (c & ~1) + 2;  // smallest even chunk index > c
                int cn = 0x7fffffff;         // next event chunk of this row
                const unsigned later = lane < 31 ? bits >> (lane + 1) : 0u;
                if (later) {
                    cn = c + 1 + __ffs(later) - 1;
                } else {
                    for (int c2 = w0 + 32; c2 < C; ++c2)
                        if (is_set(mask, i, C, c2)) { cn = c2; break; }
                }
                ref = m <= 2 * (G - 1) && m <= cn;
            }
            nref += __popc(__ballot_sync(0xffffffffu, ref));
        }
        if (lane == 0) refc[j] = nref;
    }
    __syncthreads();
    block_exclusive_scan(refc, refb, R, warp_tot);
    // 5. snapshot slots
    for (int j = warp; j < R; j += kWarps) {
        const int i = order[j];
        const int base = ptr[j];
        int run = 0, rrun = refb[j];
        for (int w0 = 0; w0 < C; w0 += 32) {
            const int c = w0 + lane;
            const bool s = c < C && is_set(mask, i, C, c);
            const unsigned bits = __ballot_sync(0xffffffffu, s);
            bool ref = false;
            if (s) {
                const int m = (c & ~1) + 2;
                int cn = 0x7fffffff;
                const unsigned later = lane < 31 ? bits >> (lane + 1) : 0u;
                if (later) {
                    cn = c + 1 + __ffs(later) - 1;
                } else {
                    for (int c2 = w0 + 32; c2 < C; ++c2)
                        if (is_set(mask, i, C, c2)) { cn = c2; break; }
                }
                ref = m <= 2 * (G - 1) && m <= cn;
            }
            const unsigned rb = __ballot_sync(0xffffffffu, ref);
            const int e = base + run + __popc(bits & ((1u << lane) - 1u));
            if (s && (int64_t)e < ev_cap) {
                const int slot = rrun + __popc(rb & ((1u << lane) - 1u));
                snap_slot[e] = ref ? slot : -1;
            }
            run += __popc(bits);
            rrun += __popc(rb);
        }
    }
    for (int j = threadIdx.x; j < R; j += kThreads) row_pair[j] = order[j];
    for (int j = threadIdx.x; j <= R; j += kThreads) row_ptr[j] = ptr[j];
    if (threadIdx.x == 0) {
        const int ns = refb[R];
        int st = 0;
        if (E > ev_cap) st |= kStatusEventOverflow;
        if (ns > snap_cap) st |= kStatusSnapOverflow;
        counts[0] = (int)E;
        counts[1] = ns;
        counts[2] = st;
        counts[3] = 0;
    }
}

}  // namespace

cudaError_t launch_select(const Problem &pb, const gdn_events &ev, int64_t snap_cap) {
    const size_t smem = sizeof(int) * (6 * (size_t)pb.R + 2);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    select_kernel<<<1, kThreads, smem, pb.stream>>>(pb.mask, pb.R, pb.C, pb.G, ev.row_pair, ev.row_ptr,
                                                    ev.ev_chunk, ev.grp_pred, ev.snap_slot, ev.counts,
                                                    (int64_t)ev.capacity, snap_cap);
    return cudaGetLastError();
}

}  // namespace gdn
