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
              int64_t snap_cap, int wait_first, int or_status, int /*part: always everything*/) {
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
// batch has few rows.  Event numbers and snapshot slots come from one pass of block
// scans over the per-word counts laid out in sorted-row order, which is CSR order.
// The kernel is bound by instruction issue on its one SM, so each word is visited
// three times only: staged, counted inside the scan, and written out.
constexpr size_t kWordsSmemLimit = 200 * 1024;

__host__ __device__ constexpr size_t words_smem_bytes(int R, int NF) {
    return sizeof(int) * (2 * (size_t)R + 3 * (size_t)NF + 2);
}

// The events of mask word w (chunks 32w..32w+31) that some group references.  By the
// snapshot rule an event at chunk c qualifies iff m = (c & ~1) + 2, the first even
// chunk after c, is at most 2(G-1) and at most the row's next event chunk.  For odd c,
// m = c + 1 and that holds for every later event; for even c it fails exactly when
// chunk c + 1, in the same word, holds an event.  So the test needs no other word.
__device__ __forceinline__ unsigned snap_bits(unsigned bits, int w, int G) {
    const int top = 2 * (G - 1) - 32 * w - 2;  // the largest allowed (c & ~1) - 32w
    const unsigned lim = top < 0 ? 0u : top >= 30 ? 0xffffffffu : (2u << ((top & ~1) + 1)) - 1u;
    return bits & (0xAAAAAAAAu | ~(bits >> 1)) & lim;
}

__device__ __forceinline__ unsigned warp_incl_scan_u(unsigned x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Exclusive scans of the words' event counts into evb[0..NF] and of their snapshot
// counts into refb[0..NF] (entry NF: the totals), word f = j*NW + w being word w of
// sorted row j.  The two counts (at most 32 each) travel packed in the halves of one
// unsigned through the warp and block steps of each 1024-word slice, whose sums stay
// below 2^16, and are unpacked into the running totals.
__device__ void word_scans(const unsigned *words, const int *order, int NW, int NF, int G, int *evb,
                           int *refb, unsigned *warp_tot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int ev_carry = 0, ref_carry = 0;
    for (int base = 0; base < NF; base += kThreads) {
        const int f = base + threadIdx.x;
        unsigned x = 0u;
        if (f < NF) {
            const int j = f / NW, w = f - j * NW;
            const unsigned bits = words[order[j] * NW + w];
            x = (unsigned)__popc(bits) | ((unsigned)__popc(snap_bits(bits, w, G)) << 16);
        }
        const unsigned incl = warp_incl_scan_u(x);
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const unsigned t = warp_tot[lane];
            const unsigned ti = warp_incl_scan_u(t);
            warp_tot[lane] = ti - t;  // exclusive warp offsets
            if (lane == 31) warp_tot[32] = ti;
        }
        __syncthreads();
        const unsigned ex = warp_tot[warp] + incl - x;
        if (f < NF) {
            evb[f] = ev_carry + (int)(ex & 0xFFFFu);
            refb[f] = ref_carry + (int)(ex >> 16);
        }
        const unsigned tot = warp_tot[32];
        ev_carry += (int)(tot & 0xFFFFu);
        ref_carry += (int)(tot >> 16);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        evb[NF] = ev_carry;
        refb[NF] = ref_carry;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
select_words_kernel(const uint8_t *__restrict__ mask, int R, int C, int G,
                    int32_t *__restrict__ row_pair, int32_t *__restrict__ row_ptr,
                    int32_t *__restrict__ ev_chunk, int32_t *__restrict__ grp_pred,
                    int32_t *__restrict__ snap_slot, int32_t *__restrict__ counts,
                    int32_t *__restrict__ run_first, int NR, int64_t ev_cap,
                    int64_t snap_cap, int wait_first, int or_status, int part) {
    extern __shared__ int sm[];
    const int NW = (C + 31) >> 5;
    const int NF = R * NW;
    int *cnt = sm;                 // [R]     events per physical row
    int *order = cnt + R;          // [R]     physical id of sorted row j
    int *evb = order + R;          // [NF+1]  first event number of word f (f = j*NW + w), then E
    int *refb = evb + NF + 1;      // [NF+1]  first snapshot slot of word f, then the slot count
    unsigned *words = reinterpret_cast<unsigned *>(refb + NF + 1);  // [NF] mask bits, physical-row major
    __shared__ unsigned warp_tot[33];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    for (int i = threadIdx.x; i < R; i += kThreads) cnt[i] = 0;
    // An online selection writes the mask just before: wait for it.  A caller's mask needs no
    // wait, so the compaction overlaps the kernel before and waits only before it exits.
    if (wait_first) pdl_wait();
    pdl_trigger();
    __syncthreads();
    // 1. stage the mask and count each row's events: one warp per (row, 256 chunks),
    //    eight coalesced loads in flight
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
        int n = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const unsigned bits = __ballot_sync(0xffffffffu, v[q]);
            const int w = 8 * b + q;
            n += __popc(bits);
            if (lane == 0 && w < NW) words[i * NW + w] = bits;
        }
        if (lane == 0) atomicAdd(&cnt[i], n);
    }
    __syncthreads();
    // 2. rank rows: count descending, id ascending
    for (int i = threadIdx.x; i < R; i += kThreads) {
        const int ci = cnt[i];
        int rank = 0;
        for (int j = 0; j < R; ++j) {
            const int cj = cnt[j];
            rank += (cj > ci) || (cj == ci && j < i);
        }
        order[rank] = i;
    }
    __syncthreads();
    if (part == 1) {  // the row order alone: the launches that need only it may start
        for (int j = threadIdx.x; j < R; j += kThreads) row_pair[j] = order[j];
        if (!wait_first) pdl_wait();
        return;
    }
    // 3. event numbers and snapshot slots of every word
    word_scans(words, order, NW, NF, G, evb, refb, warp_tot);
    // 4. one warp per (sorted row j, word w), lane = chunk 32w + lane: event chunks and
    //    snapshot slots, run starts and group predecessors
    for (int f = warp; f < NF; f += kWarps) {
        const int j = f / NW, w = f - j * NW;
        const int i = order[j];
        const unsigned bits = words[i * NW + w];
        const int e0 = evb[f];
        if (run_first && lane < 2) {  // runs of 16 chunks starting inside this word
            const int rr = 2 * w + lane;
            if (rr < NR) run_first[(int64_t)j * (NR + 1) + rr] = e0 + (lane ? __popc(bits & 0xFFFFu) : 0);
        }
        if (lane < 16) {  // groups r with 2r = 32w + 2 lane
            const int r = 16 * w + lane;
            if (r < G) {
                const int n_before = e0 + __popc(bits & ((1u << (2 * lane)) - 1u));
                grp_pred[(int64_t)i * G + r] = n_before > evb[j * NW] ? n_before - 1 : -1;
            }
        }
        if ((bits >> lane) & 1u) {
            const int e = e0 + __popc(bits & below);
            if ((int64_t)e < ev_cap) {
                const unsigned rb = snap_bits(bits, w, G);
                ev_chunk[e] = 32 * w + lane;
                snap_slot[e] = ((rb >> lane) & 1u) ? refb[f] + __popc(rb & below) : -1;
            }
        }
    }
    for (int j = threadIdx.x; j < R; j += kThreads) {
        if (part == 0) row_pair[j] = order[j];
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
                          bool wait_first, bool or_status, int part) {
    const int NW = (pb.C + 31) / 32, NR = (pb.C + kRunChunks - 1) / kRunChunks;
    const size_t fast = words_smem_bytes(pb.R, pb.R * NW);
    const bool use_words = fast <= kWordsSmemLimit;
    if (!use_words && part == 2) return cudaSuccess;  // part 1 did everything
    if (!use_words) part = 0;
    auto kernel = use_words ? select_words_kernel : select_kernel;
    const size_t smem = use_words ? fast : sizeof(int) * (6 * (size_t)pb.R + 2 + (size_t)kWarps * NW);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(pb.pdl, kernel, 1, kThreads, smem, pb.stream, pb.mask, pb.R, pb.C, pb.G, ev.row_pair,
                         ev.row_ptr, ev.ev_chunk, ev.grp_pred, ev.snap_slot, ev.counts, run_first, NR,
                         (int64_t)ev.capacity, snap_cap, (int)wait_first, (int)or_status, part);
}

}  // namespace gdn
