// sched.cu - device-side varlen scheduler.
//
// Reads query_lengths / kv_lengths on the device (they never go to the
// host), validates them, and for prefill writes the list of work items
// (batch, query block of item_tokens tokens, KV head, cost) sorted by cost, longest first, so that
// the persistent prefill grid starts the biggest items first.  Cost is the
// number of 128-key tiles the item visits after causal and length
// skipping.  For decode it only validates and clears the split tickets.
//
// Work-list layout in the workspace: int n_items at byte 0, int4 items from
// byte WS_HEADER.  On bad lengths it writes RGA_ERR_DEVICE_LENGTHS (4) to
// the status word and an empty list, so no attention work runs.
#include "device_common.cuh"
#include "kernels.h"

namespace rga {

constexpr int SCHED_THREADS = 1024;
constexpr int COST_BUCKETS = 1024;
static_assert(COST_BUCKETS == SCHED_THREADS, "one bucket per thread in the scan");

__device__ __forceinline__ int item_cost(const AttnParams &p, const SeqInfo &s, int qt) {
    int i_last = min((qt + 1) * p.item_tokens, s.q_len) - 1;
    int n = key_extent(p.causal, i_last, s);
    int c = (n + BN - 1) / BN;
    return c;
}

__global__ void __launch_bounds__(SCHED_THREADS)
sched_kernel(AttnParams p, int decode) {
    __shared__ int hist[COST_BUCKETS];
    __shared__ int bad;
    __shared__ int total;
    int *hdr = reinterpret_cast<int *>(p.ws);
    int4 *items = reinterpret_cast<int4 *>(p.ws + WS_HEADER);
    const int tid = threadIdx.x;

    if (tid == 0) { bad = 0; total = 0; }
    for (int c = tid; c < COST_BUCKETS; c += SCHED_THREADS) hist[c] = 0;
    __syncthreads();

    // 1. validate lengths, count items per cost bucket
    for (int b = tid; b < p.B; b += SCHED_THREADS) {
        const int32_t *ql = p.query_lengths, *kl = p.kv_lengths;
        SeqInfo s = seq_info(p, b);
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
        if (!ok) { atomicOr(&bad, 1); continue; }
        if (decode) continue;
        const int nqt = (s.q_len + p.item_tokens - 1) / p.item_tokens;
        for (int qt = 0; qt < nqt; ++qt) {
            int c = min(item_cost(p, s, qt), COST_BUCKETS - 1);
            atomicAdd(&hist[c], p.Hkv);
            atomicAdd(&total, p.Hkv);
        }
    }
    __syncthreads();
    if (bad || total > p.max_items) {
        if (tid == 0) {
            set_status(p.status, 4);
            hdr[0] = 0;
            hdr[1] = 0;
            hdr[2] = 0;
        }
        return;
    }

    if (decode) {
        // clear the per-(batch, kv head) split tickets and list the decode
        // units (batch, KV head, split, splits of the pair)
        int *tickets = reinterpret_cast<int *>(p.ws + WS_HEADER);
        for (int i = tid; i < p.B * p.Hkv; i += SCHED_THREADS) tickets[i] = 0;
        int4 *units = reinterpret_cast<int4 *>(p.ws + dec_units_off(p));
        for (int b = tid; b < p.B; b += SCHED_THREADS) {
            const SeqInfo s = seq_info(p, b);
            const int rows = s.q_len * p.G;
            if (rows <= 0) continue;
            const int ns = dec_splits(p, s);
            const int pos = atomicAdd(&total, ns * p.Hkv);
            for (int sp = 0; sp < ns; ++sp)
                for (int g = 0; g < p.Hkv; ++g)
                    units[pos + sp * p.Hkv + g] = make_int4(b, g, sp, ns);
        }
        __syncthreads();
        if (tid == 0) {
            hdr[0] = total;   // units listed (0 also when nothing to do)
            hdr[1] = 0;       // next unit to take
            hdr[2] = 1;       // lengths accepted
        }
        return;
    }

    // 2. bucket starts, largest cost first: exclusive block scan, thread t
    //    owning bucket COST_BUCKETS-1-t
    {
        __shared__ int warp_sum[SCHED_THREADS / 32];
        const int c = COST_BUCKETS - 1 - tid, lane = tid & 31, w = tid >> 5;
        const int h = hist[c];
        int x = h;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[w] = x;
        __syncthreads();
        if (w == 0) {
            int s = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sum[lane] = s;   // inclusive prefix over warps
        }
        __syncthreads();
        const int before = (w > 0 ? warp_sum[w - 1] : 0) + x - h;
        hist[c] = before;
        if (tid == SCHED_THREADS - 1) {
            hdr[0] = before + h;
            hdr[1] = 0;
        }
    }
    __syncthreads();

    // 3. scatter items into their sorted positions
    for (int b = tid; b < p.B; b += SCHED_THREADS) {
        SeqInfo s = seq_info(p, b);
        const int nqt = (s.q_len + p.item_tokens - 1) / p.item_tokens;
        for (int qt = nqt - 1; qt >= 0; --qt) {
            int cost = item_cost(p, s, qt);
            int c = min(cost, COST_BUCKETS - 1);
            int pos = atomicAdd(&hist[c], p.Hkv);
            for (int g = 0; g < p.Hkv; ++g) items[pos + g] = make_int4(b, qt, g, cost);
        }
    }
}

cudaError_t launch_sched(const AttnParams &p, int decode, cudaStream_t s) {
    sched_kernel<<<1, SCHED_THREADS, 0, s>>>(p, decode);
    return cudaGetLastError();
}

}  // namespace rga
