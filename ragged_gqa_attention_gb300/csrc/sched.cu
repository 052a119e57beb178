// sched.cu - device-side varlen scheduler.
//
// Reads query_lengths / kv_lengths on the device (they never go to the
// host), validates them, and for prefill writes the list of work items
// (batch, query block of item_tokens tokens, KV head, cost) sorted by cost, longest first, so that
// the persistent prefill grid starts the biggest items first.  Cost is the
// number of 128-key tiles the item visits after causal and length
// skipping.  (The decode kernel validates and lists its own work.)
//
// Work-list layout in the workspace: int n_items at byte 0, the attention
// kernel's next-item counter (cleared here) at byte 4, int4 items from
// byte WS_HEADER.  On bad lengths it writes RGA_ERR_DEVICE_LENGTHS (4) to
// the status word and an empty list, so no attention work runs; the same
// for a page index outside the pools of a paged cache.
#include "device_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace rga {

#ifndef RGA_SCHED_THREADS
#define RGA_SCHED_THREADS 256
#endif
constexpr int SCHED_THREADS = RGA_SCHED_THREADS;
constexpr int COST_BUCKETS = SCHED_THREADS;
constexpr int SCHED_MAX_B = 4096;   // per-batch prefix in shared memory up to this batch
static_assert(COST_BUCKETS == SCHED_THREADS, "one bucket per thread in the scan");

__device__ __forceinline__ int item_cost(const AttnParams &p, const SeqInfo &s, int qt) {
    int i_last = min((qt + 1) * p.item_tokens, s.q_len) - 1;
    int n = key_extent(p.causal, i_last, s);
    int c = (n + BN - 1) / BN;
    return c;
}

// Block-wide exclusive scan of one int per thread (all SCHED_THREADS threads
// call it); returns this thread's prefix and sets *total to the block sum.
__device__ __forceinline__ int block_excl_scan(int x, int *warp_sum, int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) warp_sum[w] = v;
    __syncthreads();
    if (w == 0) {
        int t = lane < SCHED_THREADS / 32 ? warp_sum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_sum[lane] = t;
    }
    __syncthreads();
    const int before = (w > 0 ? warp_sum[w - 1] : 0) + v - x;
    *total = warp_sum[SCHED_THREADS / 32 - 1];   // every thread: the block total
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(SCHED_THREADS)
sched_kernel(AttnParams p, int decode) {
    __shared__ int hist[COST_BUCKETS];
    __shared__ int qoff[SCHED_MAX_B + 1];    // per-batch first query block
    __shared__ int warp_sum[32];
    __shared__ int bad;
    __shared__ int total;
    __shared__ int nblocks;
    int *hdr = reinterpret_cast<int *>(p.ws);
    int4 *items = reinterpret_cast<int4 *>(p.ws + WS_HEADER);
    const int tid = threadIdx.x;

    pdl_launch_dependents();   // the attention kernel may start its prologue
    if (tid == 0) { bad = 0; total = 0; nblocks = 0; }
    for (int c = tid; c < COST_BUCKETS; c += SCHED_THREADS) hist[c] = 0;
    __syncthreads();

    // 1. validate lengths
    for (int b = tid; b < p.B; b += SCHED_THREADS) {
        const int32_t *ql = p.query_lengths, *kl = p.kv_lengths;
        const SeqInfo s = seq_info(p, b);
        bool ok = s.q_len >= 0 && s.kv_len >= 0;
        if (ql) ok = ok && ql[0] == 0;
        if (p.q_packed) ok = ok && ql[b + 1] <= p.q_seq;
        else ok = ok && s.q_len <= p.q_seq;
        if (p.kv_packed) ok = ok && kl[0] == 0 && kl[b + 1] <= p.kv_seq;
        else ok = ok && s.kv_len <= p.kv_seq;
        if (p.mask) {
            if (p.md[2] != 1 && p.md[2] < s.q_len) ok = false;
            if (p.md[3] != 1 && p.md[3] < s.kv_len) ok = false;
        }
        if (!ok) atomicOr(&bad, 1);
    }
    // a paged cache: every page index a sequence's keys use must lie in the
    // pools (entries past the last page are never read)
    if (p.paged) {
        const long long total = (long long)p.B * p.max_pages;
        const long long cap = (long long)p.max_pages * p.page_size;
        for (long long i = tid; i < total; i += SCHED_THREADS) {
            const int b = (int)(i / p.max_pages), k = (int)(i % p.max_pages);
            const long long len = min((long long)max(p.kv_lengths[b], 0), cap);
            if (k >= (len + p.page_size - 1) / p.page_size) continue;
            const int32_t *pt = p.page_table + (size_t)b * 2 * p.max_pages;
            const int a = pt[k], v = pt[p.max_pages + k];
            if (a < 0 || a >= p.num_pages || v < 0 || v >= p.num_pages) atomicOr(&bad, 1);
        }
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            set_status(p.status, 4);
            hdr[0] = 0;
            hdr[1] = 0;
            hdr[2] = 0;
        }
        return;
    }

    // 2. query blocks per batch and their prefix (batch-parallel)
    const bool par = p.B <= SCHED_MAX_B;
    if (par) {
        for (int base = 0; base < p.B; base += SCHED_THREADS) {
            const int b = base + tid;
            int n = 0;
            if (b < p.B) {
                const SeqInfo s = seq_info(p, b);
                n = (s.q_len + p.item_tokens - 1) / p.item_tokens;
            }
            int chunk_total;
            const int before = block_excl_scan(n, warp_sum, &chunk_total);
            if (b < p.B) qoff[b] = nblocks + before;
            __syncthreads();
            if (tid == 0) nblocks += chunk_total;
            __syncthreads();
        }
        if (tid == 0) qoff[p.B] = nblocks;
        __syncthreads();
    }

    // (batch, query block) of flat block index i
    auto locate = [&](int i, int &b, int &qt) {
        int lo = 0, hi = p.B;                 // qoff[lo] <= i < qoff[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (qoff[mid] <= i) lo = mid; else hi = mid;
        }
        b = lo;
        qt = i - qoff[lo];
    };

    // 3. cost histogram
    if (par) {
        for (int i = tid; i < nblocks; i += SCHED_THREADS) {
            int b, qt;
            locate(i, b, qt);
            const SeqInfo s = seq_info(p, b);
            atomicAdd(&hist[min(item_cost(p, s, qt), COST_BUCKETS - 1)], p.Hkv);
        }
        if (tid == 0) total = nblocks * p.Hkv;
    } else {
        for (int b = tid; b < p.B; b += SCHED_THREADS) {
            const SeqInfo s = seq_info(p, b);
            const int nqt = (s.q_len + p.item_tokens - 1) / p.item_tokens;
            for (int qt = 0; qt < nqt; ++qt) {
                atomicAdd(&hist[min(item_cost(p, s, qt), COST_BUCKETS - 1)], p.Hkv);
                atomicAdd(&total, p.Hkv);
            }
        }
    }
    __syncthreads();
    if (total > p.max_items) {
        if (tid == 0) {
            set_status(p.status, 4);
            hdr[0] = 0;
            hdr[1] = 0;
        }
        return;
    }

    // 4. bucket starts, largest cost first: thread t owns bucket COST_BUCKETS-1-t
    {
        const int c = COST_BUCKETS - 1 - tid;
        const int h = hist[c];
        int all;
        const int before = block_excl_scan(h, warp_sum, &all);
        hist[c] = before;
        if (tid == 0) {
            hdr[0] = all;
            hdr[1] = 0;
        }
    }
    __syncthreads();

    // 5. scatter items into their sorted positions
    if (par) {
        for (int i = tid; i < nblocks; i += SCHED_THREADS) {
            int b, qt;
            locate(i, b, qt);
            const SeqInfo s = seq_info(p, b);
            const int cost = item_cost(p, s, qt);
            const int pos = atomicAdd(&hist[min(cost, COST_BUCKETS - 1)], p.Hkv);
            for (int g = 0; g < p.Hkv; ++g)
                if (dbg_ok(pos + g < p.max_items, p.status))
                    items[pos + g] = make_int4(b, qt, g, cost);
        }
    } else {
        for (int b = tid; b < p.B; b += SCHED_THREADS) {
            const SeqInfo s = seq_info(p, b);
            const int nqt = (s.q_len + p.item_tokens - 1) / p.item_tokens;
            for (int qt = nqt - 1; qt >= 0; --qt) {
                const int cost = item_cost(p, s, qt);
                const int pos = atomicAdd(&hist[min(cost, COST_BUCKETS - 1)], p.Hkv);
                for (int g = 0; g < p.Hkv; ++g)
                    if (dbg_ok(pos + g < p.max_items, p.status))
                        items[pos + g] = make_int4(b, qt, g, cost);
            }
        }
    }
}

cudaError_t launch_sched(const AttnParams &p, int decode, cudaStream_t s) {
    sched_kernel<<<1, SCHED_THREADS, 0, s>>>(p, decode);
    return cudaGetLastError();
}

}  // namespace rga
