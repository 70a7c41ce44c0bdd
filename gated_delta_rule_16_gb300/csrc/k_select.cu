// k_select.cu -- event compaction: [B,P,C] mask -> CSR event lists
// (SparseGDN Sec. 2.5, Eq. 16: rows per head pair, events in time order,
// per-group predecessor event, device-resident event count).
//
// One CTA of 1024 threads does the whole batch: the mask is tiny (B*P*C bytes,
// 8 KiB at T = 32K) and the work is integer bookkeeping, so a single CTA with
// warp ballots and block scans keeps it to a few microseconds and bit-exact.
// Two variants: a word-parallel one for masks that fit in shared memory as bit
// words (the usual case), and a row-per-warp one for larger batches.
//
// Row order: event count descending, ties by physical row id ascending.
// Snapshot rule: event e (chunk c, next event of its row at chunk cn, or none)
// is some group's predecessor iff an even chunk index 2r with c < 2r <= cn
// exists and 2r <= 2(G-1); such events are numbered densely in event order.
#include <climits>

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

// One warp stages the 0/1 bits of mask row `row` as 32-chunk words: the loads of
// 512 chunks are issued together before the ballots (mask == NULL: all chunks set).
__device__ __forceinline__ void stage_row(const uint8_t *__restrict__ mask, int64_t row, int C, int NW,
                                          unsigned *wrow) {
    const int lane = threadIdx.x & 31;
    const uint8_t *mr = mask ? mask + row * C : nullptr;
    for (int c0 = 0; c0 < C; c0 += 512) {
        bool v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int c = c0 + 32 * q + lane;
            v[q] = c < C && (mr == nullptr || mr[c] != 0);
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const unsigned bits = __ballot_sync(0xffffffffu, v[q]);
            const int w = (c0 >> 5) + q;
            if (lane == 0 && w < NW) wrow[w] = bits;
        }
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kThreads)
select_kernel(const uint8_t *__restrict__ mask, int R, int C, int G,
              int32_t *__restrict__ row_pair, int32_t *__restrict__ row_ptr,
              int32_t *__restrict__ ev_chunk, int32_t *__restrict__ grp_pred,
              int32_t *__restrict__ snap_slot, int32_t *__restrict__ counts,
              int32_t *__restrict__ run_first, int NR, int64_t ev_cap,
              int64_t snap_cap, int wait_first, int or_status) {
    extern __shared__ int sm[];
    const int NW = (C + 31) >> 5;   // 32-chunk mask words per row
    int *cnt = sm;               // [R]   events per physical row
    int *order = cnt + R;        // [R]   physical id of sorted row j
    int *sorted_cnt = order + R; // [R]
    int *ptr = sorted_cnt + R;   // [R+1] row offsets
    int *refc = ptr + R + 1;     // [R]   referenced events per sorted row
    int *refb = refc + R;        // [R+1] snapshot base per sorted row
    unsigned *words = reinterpret_cast<unsigned *>(refb + R + 1);  // [kWarps][NW] one row's mask bits
    __shared__ int warp_tot[33];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // An online selection writes the mask just before: wait for it.  A caller's mask needs no
    // wait, so the compaction overlaps the kernel before and waits only before it exits.
    if (wait_first) pdl_wait();
    pdl_trigger();
    unsigned *wrow = words + warp * NW;

    // 1. events per row
    for (int i = warp; i < R; i += kWarps) {
        int n = 0;
        if (mask) {
            const uint8_t *mr = mask + (int64_t)i * C;
#pragma unroll 8
            for (int c = lane; c < C; c += 32) n += mr[c] != 0;
        } else {
            n = C > lane ? (C - lane + 31) / 32 : 0;
        }
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
    // 4. per row (one warp): stage the mask bits, write event chunks, run starts, each
    //    group's predecessor, and count the events some group references
    //    (event at chunk c, next event of the row at cn or none: referenced iff the
    //    smallest even chunk index m > c satisfies m <= cn and m <= 2(G-1)).
    for (int j = warp; j < R; j += kWarps) {
        const int i = order[j];
        const int base = ptr[j];
        stage_row(mask, i, C, NW, wrow);
        int run = 0, nref = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = 32 * w + lane;
            const unsigned bits = wrow[w];
            const bool s = (bits >> lane) & 1u;
            const int before = __popc(bits & ((1u << lane) - 1u));
            const int e = base + run + before;
            if (s && (int64_t)e < ev_cap) ev_chunk[e] = c;
            if (run_first && lane < 2) {  // runs of 16 chunks starting inside this word
                const int rr = 2 * w + lane;
                if (rr < NR) run_first[(int64_t)j * (NR + 1) + rr] = base + run + (lane ? __popc(bits & 0xFFFFu) : 0);
            }
            if (lane < 16) {  // groups r with 2r = 32w + 2 lane
                const int r = 16 * w + lane;
                if (r < G) {
                    const int n_before = run + __popc(bits & ((1u << (2 * lane)) - 1u));
                    grp_pred[(int64_t)i * G + r] = n_before > 0 ? base + n_before - 1 : -1;
                }
            }
            bool ref = false;
            if (s) {
                const int m = (c & ~1) + 2;
                int cn = 0x7fffffff;
                const unsigned later = lane < 31 ? bits >> (lane + 1) : 0u;
                if (later) {
                    cn = c + __ffs(later);
                } else {
                    for (int w2 = w + 1; w2 < NW; ++w2)
                        if (wrow[w2]) { cn = 32 * w2 + __ffs(wrow[w2]) - 1; break; }
                }
                ref = m <= 2 * (G - 1) && m <= cn;
            }
            nref += __popc(__ballot_sync(0xffffffffu, ref));
            run += __popc(bits);
        }
        if (lane == 0) {
            refc[j] = nref;
            if (run_first) run_first[(int64_t)j * (NR + 1) + NR] = base + run;
        }
        __syncwarp();
    }
    __syncthreads();
    block_exclusive_scan(refc, refb, R, warp_tot);
    // 5. snapshot slots (the row's bits are staged again)
    for (int j = warp; j < R; j += kWarps) {
        const int i = order[j];
        const int base = ptr[j];
        stage_row(mask, i, C, NW, wrow);
        int run = 0, rrun = refb[j];
        for (int w = 0; w < NW; ++w) {
            const int c = 32 * w + lane;
            const unsigned bits = wrow[w];
            const bool s = (bits >> lane) & 1u;
            bool ref = false;
            if (s) {
                const int m = (c & ~1) + 2;
                int cn = 0x7fffffff;
                const unsigned later = lane < 31 ? bits >> (lane + 1) : 0u;
                if (later) {
                    cn = c + __ffs(later);
                } else {
                    for (int w2 = w + 1; w2 < NW; ++w2)
                        if (wrow[w2]) { cn = 32 * w2 + __ffs(wrow[w2]) - 1; break; }
                }
                ref = m <= 2 * (G - 1) && m <= cn;
            }
            const unsigned rb = __ballot_sync(0xffffffffu, ref);
            const int e = base + run + __popc(bits & ((1u << lane) - 1u));
            if (s && (int64_t)e < ev_cap) snap_slot[e] = ref ? rrun + __popc(rb & ((1u << lane) - 1u)) : -1;
            run += __popc(bits);
            rrun += __popc(rb);
        }
        __syncwarp();
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
        if (or_status) atomicOr(&counts[2], st);  // other kernels of the prefill latch theirs there too
        else counts[2] = st;
        counts[3] = 0;
    }
    if (!wait_first) pdl_wait();  // this grid's completion implies its predecessors'
}

// Word-parallel variant, used when the whole mask fits in shared memory as
// 32-chunk words (B*P*ceil(C/32) words, 8 KiB of them at B = 8, T = 32K).  Every
// (sorted row, word) pair is one warp task, so all 32 warps work even when the
// batch has few rows; event numbers and snapshot slots come from block scans
// over the per-word counts laid out in sorted-row order, which is CSR order.
constexpr size_t kWordsSmemLimit = 200 * 1024;

__host__ __device__ constexpr size_t words_smem_bytes(int R, int NF) {
    return sizeof(int) * (2 * (size_t)R + 5 * (size_t)NF + 2);
}

__global__ void __launch_bounds__(kThreads)
select_words_kernel(const uint8_t *__restrict__ mask, int R, int C, int G,
                    int32_t *__restrict__ row_pair, int32_t *__restrict__ row_ptr,
                    int32_t *__restrict__ ev_chunk, int32_t *__restrict__ grp_pred,
                    int32_t *__restrict__ snap_slot, int32_t *__restrict__ counts,
                    int32_t *__restrict__ run_first, int NR, int64_t ev_cap,
                    int64_t snap_cap, int wait_first, int or_status) {
    extern __shared__ int sm[];
    const int NW = (C + 31) >> 5;
    const int NF = R * NW;
    int *cnt = sm;                 // [R]     events per physical row
    int *order = cnt + R;          // [R]     physical id of sorted row j
    int *evb = order + R;          // [NF+1]  first event number of word f (f = j*NW + w), then E
    int *refb = evb + NF + 1;      // [NF+1]  first snapshot slot of word f, then the slot count
    unsigned *words = reinterpret_cast<unsigned *>(refb + NF + 1);  // [NF] mask bits, physical-row major
    int *nxt = reinterpret_cast<int *>(words + NF);                 // [NF] first event chunk at or after word w
    unsigned *refbits = reinterpret_cast<unsigned *>(nxt + NF);     // [NF] referenced events of word f
    __shared__ int warp_tot[33];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    // An online selection writes the mask just before: wait for it.  A caller's mask needs no
    // wait, so the compaction overlaps the kernel before and waits only before it exits.
    if (wait_first) pdl_wait();
    pdl_trigger();
    // 1. stage the mask: one warp per (row, 256 chunks), eight coalesced loads in flight
    const int NB = (NW + 7) >> 3;
    for (int t = warp; t < R * NB; t += kWarps) {
        const int i = t / NB, b = t - i * NB;
        const uint8_t *mr = mask ? mask + (int64_t)i * C : nullptr;
        bool v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int c = 256 * b + 32 * q + lane;
            v[q] = c < C && (mr == nullptr || mr[c] != 0);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const unsigned bits = __ballot_sync(0xffffffffu, v[q]);
            const int w = 8 * b + q;
            if (lane == 0 && w < NW) words[i * NW + w] = bits;
        }
    }
    __syncthreads();
    // 2. per physical row: its event count and, per word, the first event chunk at or
    //    after that word (a suffix minimum, INT_MAX when the rest of the row is empty)
    for (int i = warp; i < R; i += kWarps) {
        int n = 0, carry = INT_MAX;
        for (int w0 = ((NW - 1) >> 5) << 5; w0 >= 0; w0 -= 32) {
            const int w = w0 + lane;
            const unsigned bits = w < NW ? words[i * NW + w] : 0u;
            n += __popc(bits);
            int x = bits ? 32 * w + __ffs(bits) - 1 : INT_MAX;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_down_sync(0xffffffffu, x, o);
                if (lane + o < 32) x = min(x, y);
            }
            x = min(x, carry);
            if (w < NW) nxt[i * NW + w] = x;
            carry = __shfl_sync(0xffffffffu, x, 0);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        if (lane == 0) cnt[i] = n;
    }
    __syncthreads();
    // 3. rank rows: count descending, id ascending
    for (int i = threadIdx.x; i < R; i += kThreads) {
        int ci = cnt[i], rank = 0;
        for (int j = 0; j < R; ++j) {
            int cj = cnt[j];
            rank += (cj > ci) || (cj == ci && j < i);
        }
        order[rank] = i;
    }
    __syncthreads();
    // 4. per-word event counts in sorted-row order; their exclusive scan numbers the events
    for (int f = threadIdx.x; f < NF; f += kThreads) {
        const int j = f / NW, w = f - j * NW;
        evb[f] = __popc(words[order[j] * NW + w]);
    }
    __syncthreads();
    block_exclusive_scan(evb, evb, NF, warp_tot);
    // 5. one warp per (sorted row j, word w): event chunks, run starts, group
    //    predecessors, and which events some group references (event at
    //    chunk c, next event of the row at cn or none: referenced iff the smallest even
    //    chunk index m > c satisfies m <= cn and m <= 2(G-1))
    for (int f = warp; f < NF; f += kWarps) {
        const int j = f / NW, w = f - j * NW;
        const int i = order[j];
        const unsigned bits = words[i * NW + w];
        const int e0 = evb[f], row0 = evb[j * NW];
        const int c = 32 * w + lane;
        const bool s = (bits >> lane) & 1u;
        const int e = e0 + __popc(bits & below);
        if (s && (int64_t)e < ev_cap) ev_chunk[e] = c;
        if (run_first && lane < 2) {  // runs of 16 chunks starting inside this word
            const int rr = 2 * w + lane;
            if (rr < NR) run_first[(int64_t)j * (NR + 1) + rr] = e0 + (lane ? __popc(bits & 0xFFFFu) : 0);
        }
        if (lane < 16) {  // groups r with 2r = 32w + 2 lane
            const int r = 16 * w + lane;
            if (r < G) {
                const int n_before = e0 + __popc(bits & ((1u << (2 * lane)) - 1u));
                grp_pred[(int64_t)i * G + r] = n_before > row0 ? n_before - 1 : -1;
            }
        }
        bool ref = false;
        if (s) {
            const int m = (c & ~1) + 2;
            const unsigned later = lane < 31 ? bits >> (lane + 1) : 0u;
            const int cn = later ? c + __ffs(later) : (w + 1 < NW ? nxt[i * NW + w + 1] : INT_MAX);
            ref = m <= 2 * (G - 1) && m <= cn;
        }
        const unsigned rb = __ballot_sync(0xffffffffu, ref);
        if (lane == 0) {
            refbits[f] = rb;
            refb[f] = __popc(rb);
        }
    }
    __syncthreads();
    block_exclusive_scan(refb, refb, NF, warp_tot);
    // 6. snapshot slots: referenced events numbered densely in event order
    for (int f = warp; f < NF; f += kWarps) {
        const int j = f / NW, w = f - j * NW;
        const unsigned bits = words[order[j] * NW + w];
        if (bits == 0u) continue;  // warp-uniform
        const unsigned rb = refbits[f];
        const int e = evb[f] + __popc(bits & below);
        if (((bits >> lane) & 1u) && (int64_t)e < ev_cap)
            snap_slot[e] = ((rb >> lane) & 1u) ? refb[f] + __popc(rb & below) : -1;
    }
    for (int j = threadIdx.x; j < R; j += kThreads) {
        row_pair[j] = order[j];
        if (run_first) run_first[(int64_t)j * (NR + 1) + NR] = evb[(j + 1) * NW];
    }
    for (int j = threadIdx.x; j <= R; j += kThreads) row_ptr[j] = evb[j * NW];
    if (threadIdx.x == 0) {
        const int E = evb[NF], ns = refb[NF];
        int st = 0;
        if ((int64_t)E > ev_cap) st |= kStatusEventOverflow;
        if (ns > snap_cap) st |= kStatusSnapOverflow;
        counts[0] = E;
        counts[1] = ns;
        if (or_status) atomicOr(&counts[2], st);  // other kernels of the prefill latch theirs there too
        else counts[2] = st;
        counts[3] = 0;
    }
    if (!wait_first) pdl_wait();  // this grid's completion implies its predecessors'
}

}  // namespace

cudaError_t launch_select(const Problem &pb, const gdn_events &ev, int64_t snap_cap, int32_t *run_first,
                          bool wait_first, bool or_status) {
    const int NW = (pb.C + 31) / 32, NR = (pb.C + kRunChunks - 1) / kRunChunks;
    const size_t fast = words_smem_bytes(pb.R, pb.R * NW);
    const bool use_words = fast <= kWordsSmemLimit;
    auto kernel = use_words ? select_words_kernel : select_kernel;
    const size_t smem = use_words ? fast : sizeof(int) * (6 * (size_t)pb.R + 2 + (size_t)kWarps * NW);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(pb.pdl, kernel, 1, kThreads, smem, pb.stream, pb.mask, pb.R, pb.C, pb.G, ev.row_pair,
                         ev.row_ptr, ev.ev_chunk, ev.grp_pred, ev.snap_slot, ev.counts, run_first, NR,
                         (int64_t)ev.capacity, snap_cap, (int)wait_first, (int)or_status);
}

}  // namespace gdn
