// prefill.cuh - fused attention forward for sm_103a on the 5th-generation
// tensor cores (tcgen05 + TMEM), with TMA-staged, 128-byte-swizzled Q/K/V
// tiles and warp-specialised roles.
//
// Computes, per work item (batch b, KV head g, two query tiles):
//   S = Q K^T (BMM1, fp32 in TMEM)  ->  scale, causal / length / mask
//   ->  softmax (online, fp32, exp2) or 'none'  ->  optional fp8/int8 Q/DQ
//   ->  O += P V (BMM2, fp32 in TMEM)  ->  O / l  ->  Y
// following "TensorRT Custom Operator Schemas" (TRT_Attention,
// TRT_QuantizedAttention) and the MHA/GQA AttentionPlugin of the "TensorRT
// Plugins Guide".
//
// GQA reuse: the 128 rows of a query tile are the G = Hq/Hkv query heads of
// one KV head times TQ = 128/G tokens, so every K/V tile is loaded once for
// the whole group.  Row r maps to (token t, head hh) as r = t*G + hh for
// packed Q ([T,H,D]: the G heads of a token are adjacent) and r = hh*TQ + t
// for padded Q ([B,H,N,D]).  A work item holds two such tiles (2*TQ tokens)
// that share every K/V tile.
//
// Roles (384 threads, three warpgroups):
//   warps 0-3  softmax warpgroup of tile 0 (thread = TMEM lane = row)
//   warps 4-7  softmax warpgroup of tile 1
//   warp 8     TMEM owner and single-thread MMA issuer
//   warp 9     TMA producer (Q once per item, K and V rings)
//   warps 10-11 idle (they only give up their registers)
// Tensor-core order per key tile j:  S0(j+1) after O0 += P0(j) V(j), and
// S1(j+1) after O1 += P1(j) V(j), so while one warpgroup turns its scores
// into probabilities the tensor core works for the other one.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P (16-bit) is written over the S columns it came from and fed to BMM2 from
// TMEM; only V is read from shared memory for BMM2.
//
// The grid is persistent (one CTA per SM); CTA c takes items c, c+grid, ...
// of the work list, which the scheduler sorted longest first.
#pragma once
#include <cuda.h>
#include <type_traits>
#include "device_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace rga {

constexpr int PF_THREADS = 384;
// Register split: the CTA is launched with PF_LAUNCH_REGS registers per
// thread (the most 384 threads can have); the MMA/TMA warpgroup then drops
// to PF_AUX_REGS and each softmax warpgroup rises to PF_SOFTMAX_REGS.
// 2 * 128 * PF_SOFTMAX_REGS + 128 * PF_AUX_REGS must not exceed
// 384 * PF_LAUNCH_REGS, or the increase would wait forever; the host checks
// the kernel's register count before it launches.
constexpr int PF_LAUNCH_REGS = 168;
constexpr int PF_SOFTMAX_REGS = 200;
constexpr int PF_AUX_REGS = 104;
static_assert(2 * 128 * PF_SOFTMAX_REGS + 128 * PF_AUX_REGS <= PF_THREADS * PF_LAUNCH_REGS,
              "register split exceeds the launch allocation");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 0, O_COL0 = 256;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units: rescale O when the max grows by > 2^8
constexpr float RESCALE_SUM = 256.0f;       // 2^RESCALE_THRESHOLD
constexpr float LOG2E = 1.4426950408889634f;

// Per-item geometry, computed identically by every role.
struct Item {
    int b, qt, g;
    SeqInfo s;
    int i0;          // first query token of the item (within the sequence)
    int ntok;        // valid tokens in the item (<= 2 * TQ)
    int nkt;         // key tiles visited
    int ntiles;      // BMM1 steps per tile (2 * nkt for the two-pass quantized softmax)
};

// Work items are handed out dynamically: a CTA's first item is its block
// index, every later one comes from a global counter (the work list's
// second header word, cleared by the scheduler), so that a CTA that drew
// short items takes more of them.  The producer warp draws the index and
// passes it to the other roles through a ring of IRING slots in shared
// memory, each slot holding the whole Item (the producer reads the work
// list and the sequence lengths; the other roles make no global loads to
// start an item).
constexpr int IRING = 4;
constexpr int ITEM_CONSUMERS = 1 + 8;   // the MMA warp and the 8 softmax warps

// KV8: K and V hold E4M3 codes (an FP8 KV cache).  The producer lands each
// 128-key tile as bytes (128 rows x D bytes, unswizzled) and the two
// converter warps expand it into the 16-bit, 128-byte-swizzled tile the
// tensor core reads.  For D = 128 the bytes land in the second 64-column
// block of the 16-bit stage itself (the expansion writes row r of a block
// only over byte row r, which the same warp has already read); for D = 64
// they land in buffers of their own.
template <int D, bool KV8 = false>
struct PfLayout {
    static constexpr int KST = D == 128 ? 2 : 3;         // K ring stages
    static constexpr int VST = D == 128 ? 2 : 3;         // V ring stages
    static constexpr int BLK = 128 * 128;                // one 64-column block of 128 rows
    static constexpr int NBLK = D / 64;
    static constexpr int TILE = NBLK * BLK;              // 128 rows x D x 2 bytes
    static constexpr int RAW_TILE = 128 * D;             // 128 rows x D bytes (KV8)
    static constexpr int Q_OFF = 0;                      // two Q tiles
    static constexpr int K_OFF = Q_OFF + 2 * TILE;
    static constexpr int V_OFF = K_OFF + KST * TILE;
    // epilogue staging: 32 rows x 128 bytes per softmax warp (8 warps)
    static constexpr int STG_OFF = V_OFF + VST * TILE;
    static constexpr int STG_WARP = 32 * 128;
    // KV8 byte tiles of their own (D = 64 only)
    static constexpr bool RAW_SEP = KV8 && D != 128;
    static constexpr int RAW_OFF = STG_OFF + 8 * STG_WARP;
    static constexpr int BAR_OFF = RAW_OFF + (RAW_SEP ? (KST + VST) * RAW_TILE : 0);
    // barriers: q_full, q_empty, k_full[KST], k_empty[KST], v_full[VST],
    // v_empty[VST], s_full[2], p_full[2], o_done[2], v_part,
    // item_full[IRING], item_empty[IRING], kraw_full[KST], vraw_full[VST],
    // q_conv
    static constexpr int NBAR = 2 + 2 * KST + 2 * VST + 7 + 2 * IRING + KST + VST + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    // misc: TMEM address (+0), abort flag (+8), the Q tiles' score factors
    // 2^s (+16, +20; FP8 cache with bf16 queries), the converter warps' Q
    // maxima (+24..+39), item ring (+64)
    static constexpr int RING_OFF = 64;
    static constexpr int BYTES = MISC_OFF + 256;
    // room to align the base to 1024; at least 120 KB so that only one CTA
    // (and one 512-column TMEM allocation) is resident per SM
    static constexpr int ALLOC = (BYTES + 1024) > 120 * 1024 ? (BYTES + 1024) : 120 * 1024;
    static_assert(ALLOC <= 232448, "shared memory per CTA");
    // byte tile of K stage s / V stage s (KV8)
    __host__ __device__ static constexpr int raw_k(int st) {
        return RAW_SEP ? RAW_OFF + st * RAW_TILE : K_OFF + st * TILE + BLK;
    }
    __host__ __device__ static constexpr int raw_v(int st) {
        return RAW_SEP ? RAW_OFF + (KST + st) * RAW_TILE : V_OFF + st * TILE + BLK;
    }
};

struct PfBars {
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *p_full,
        *o_done, *v_part, *item_full, *item_empty, *kraw_full, *vraw_full, *q_conv;
    Item *ring;   // IRING items
};

template <int D, bool KV8>
__device__ __forceinline__ PfBars pf_bars(uint8_t *base) {
    using L = PfLayout<D, KV8>;
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    PfBars r;
    r.q_full = b;
    r.q_empty = b + 1;
    r.k_full = b + 2;
    r.k_empty = r.k_full + L::KST;
    r.v_full = r.k_empty + L::KST;
    r.v_empty = r.v_full + L::VST;
    r.s_full = r.v_empty + L::VST;
    r.p_full = r.s_full + 2;
    r.o_done = r.p_full + 2;
    r.v_part = r.o_done + 2;
    r.item_full = r.v_part + 1;
    r.item_empty = r.item_full + IRING;
    r.kraw_full = r.item_empty + IRING;
    r.vraw_full = r.kraw_full + L::KST;
    r.q_conv = r.vraw_full + L::VST;
    static_assert(L::RING_OFF + IRING * sizeof(Item) <= 256, "item ring fits the misc area");
    r.ring = reinterpret_cast<Item *>(base + (L::MISC_OFF - L::BAR_OFF) + L::RING_OFF);
    return r;
}

// Consumer side of the item ring: this role's n-th item; false at the end
// of the work (an item with b < 0) or when a wait gave up.  One arrival per
// consumer (a whole softmax warp arrives once, from lane 0).
__device__ __forceinline__ bool next_item(const PfBars &bar, uint32_t n, volatile int *abort,
                                          bool warp_consumer, Item &m) {
    const int slot = n % IRING;
    if (!mbar_wait(&bar.item_full[slot], (n / IRING) & 1, abort)) return false;
    m = bar.ring[slot];
    if (warp_consumer) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&bar.item_empty[slot]);
    } else {
        mbar_arrive(&bar.item_empty[slot]);
    }
    return m.b >= 0;
}

template <int MODE>
__device__ __forceinline__ Item load_item(const AttnParams &p, int idx) {
    int4 it = make_int4(0, 0, 0, 0);   // (debug checks) inside the work list
    if (dbg_ok(idx >= 0 && idx < p.max_items, p.status))
        it = reinterpret_cast<const int4 *>(p.ws + WS_HEADER)[idx];
    Item m;
    m.b = it.x;
    m.qt = it.y;
    m.g = it.z;
    m.s = seq_info(p, m.b);
    m.i0 = m.qt * p.item_tokens;
    m.ntok = min(p.item_tokens, m.s.q_len - m.i0);
    const int n = key_extent(p.causal, m.i0 + m.ntok - 1, m.s);
    m.nkt = (n + BN - 1) / BN;
    m.ntiles = (MODE == MODE_SOFTMAX_Q) ? 2 * m.nkt : m.nkt;
    return m;
}

// Whether BMM1 step t is followed by a BMM2 (pass 1 of the two-pass
// quantized softmax only gathers row statistics).
template <int MODE>
__device__ __forceinline__ bool is_pv(const Item &m, int t) {
    return MODE != MODE_SOFTMAX_Q || t >= m.nkt;
}
template <int MODE>
__device__ __forceinline__ int key_tile(const Item &m, int t) {
    return (MODE == MODE_SOFTMAX_Q && t >= m.nkt) ? t - m.nkt : t;
}

// ------------------------------------------------------------------ loads
// After a V tile whose keys run past the sequence end (only `rem` < 128 rows
// valid) has landed, zero the rows from `rem` on (they may hold NaN, and
// 0 * NaN would reach O) and publish the change to the tensor core through
// the async proxy.  The 128-byte swizzle only permutes 16-byte chunks within
// a row, so whole rows are cleared in place.
template <int D>
__device__ void zero_v_rows(uint8_t *tile, int rem, int lane) {
    constexpr int NBLK = D / 64;
    const int first = rem < 0 ? 0 : rem;
    const int nchunks = (128 - first) * 8 * NBLK;   // 16-byte chunks to clear
    for (int idx = lane; idx < nchunks; idx += 32) {
        const int blk = idx % NBLK, rest = idx / NBLK;
        const int r = first + rest / 8, cc = rest % 8;
        *reinterpret_cast<uint4 *>(tile + blk * PfLayout<D>::BLK + r * 128 + cc * 16) =
            make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// TMA box of query tile `a` of the item (per 64-column block).
__device__ __forceinline__ void tma_q(const AttnParams &p, const CUtensorMap *map,
                                      const Item &m, int a, void *dst, uint64_t *bar, int d0) {
    const int tok = m.i0 + a * p.tq;
    if (p.q_packed)   // dims (D, Hq, T): box (64, G, TQ)
        tma_load_3d(dst, map, bar, d0, m.g * p.G, m.s.q_off + tok);
    else              // dims (D, Nq, Hq, B): box (64, TQ, G, 1)
        tma_load_4d(dst, map, bar, d0, tok, m.g * p.G, m.b);
}
__device__ __forceinline__ void tma_kv(const AttnParams &p, const CUtensorMap *map,
                                       const Item &m, int j0, void *dst, uint64_t *bar,
                                       int d0) {
    if (p.kv_packed)  // dims (D, Hkv, T): box (64, 1, 128)
        tma_load_3d(dst, map, bar, d0, m.g, m.s.kv_off + j0);
    else              // dims (D, Nkv, Hkv, B): box (64, 128, 1, 1)
        tma_load_4d(dst, map, bar, d0, j0, m.g, m.b);
}

// Pool page of each pr-row sub-box of key tile j0 of a paged cache: lane i
// (i < BN / pr) gets the page holding keys j0 + i * pr .. + pr - 1 (table
// row `which`: 0 K, 1 V), or -1 past the sequence's last page, where the
// TMA copy reads out of bounds and fills zeros.  (The scheduler checked
// every page index the sequence's keys use.)
__device__ __forceinline__ int tile_page(const AttnParams &p, const Item &m, int which, int j0,
                                         int pr) {
    const int lane = threadIdx.x & 31;
    int pg = -1;
    if (lane < BN / pr) {
        const int idx = (j0 + lane * pr) / p.page_size;
        const int npages = (m.s.kv_len + p.page_size - 1) / p.page_size;
        if (idx < npages)
            pg = __ldg(p.page_table + ((size_t)m.b * 2 + which) * p.max_pages + idx);
    }
    return pg;
}

// Key tile j0 of K (which = 0) or V (which = 1) into dst, every copy
// completing on `bar` (whose transaction count is set to `bytes`).  16-bit:
// NBLK boxes of 64 columns x 128 rows, 128-byte swizzled; KV8: one box of D
// bytes x 128 rows, unswizzled.  A paged cache takes the tile as BN / pr
// boxes of pr rows, each inside one page, whose page ids the warp's lanes
// read together.  The whole warp calls it; lane 0 issues.  (The producer's
// issue latency is on the pipeline's critical path: a linear tile is two or
// three instructions from lane 0, with no shuffles.)
template <int D, bool KV8, bool PAGED>
__device__ __forceinline__ void load_kv_tile(const AttnParams &p, const CUtensorMap *map,
                                             const Item &m, int which, int j0, uint8_t *dst,
                                             uint64_t *bar, uint32_t bytes) {
    using L = PfLayout<D, KV8>;
    const int lane = threadIdx.x & 31;
    if (!PAGED) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, bytes);
            // (debug checks) the tile starts inside the sequence and the cache
            if (!dbg_ok(j0 >= 0 && j0 < m.s.kv_len && m.g < p.Hkv &&
                        (p.kv_packed ? m.s.kv_off + j0 < p.kv_seq : j0 < p.kv_seq && m.b < p.B),
                        p.status)) {
                mbar_complete_tx(bar, bytes);
                return;
            }
            if (KV8) {
                if (p.kv_packed) tma_load_3d(dst, map, bar, 0, m.g, m.s.kv_off + j0);
                else tma_load_4d(dst, map, bar, 0, j0, m.g, m.b);
            } else {
                for (int blk = 0; blk < L::NBLK; ++blk)
                    tma_kv(p, map, m, j0, dst + blk * L::BLK, bar, blk * 64);
            }
        }
        return;
    }
    const int pr = pf_page_rows(p.page_size);
    const int mine = tile_page(p, m, which, j0, pr);
    int pg[BN / 32];
#pragma unroll
    for (int i = 0; i < BN / 32; ++i) pg[i] = __shfl_sync(0xffffffffu, mine, i);
    if (lane == 0) {
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int i = 0; i < BN / 32; ++i) {
            if (i * pr >= BN) break;
            const int key = j0 + i * pr, row = key % p.page_size;
            // (debug checks) a box in one of the sequence's pages lies in the
            // pools; boxes past its last page read out of bounds (-1)
            if (!dbg_ok(key / p.page_size >= (m.s.kv_len + p.page_size - 1) / p.page_size
                            ? pg[i] == -1 : (pg[i] >= 0 && pg[i] < p.num_pages),
                        p.status)) {
                mbar_complete_tx(bar, bytes / (BN / pr));
                continue;
            }
            if (KV8) {
                tma_load_4d(dst + i * pr * D, map, bar, 0, row, m.g, pg[i]);
            } else {
                for (int blk = 0; blk < L::NBLK; ++blk)
                    tma_load_4d(dst + blk * L::BLK + i * pr * 128, map, bar, blk * 64, row, m.g,
                                pg[i]);
            }
        }
    }
}

// PAGED: K and V come from page pools (both forms are compiled into every
// kernel and the producer picks one at the start, so the linear form's loop
// carries no page logic).
template <int D, int MODE, bool KV8, bool PAGED>
__device__ __forceinline__ void producer_role(const AttnParams &p, const TensorMaps &tm, uint8_t *sm,
                              const PfBars &bar, volatile int *abort, int n_items) {
    using L = PfLayout<D, KV8>;
    const int lane = threadIdx.x & 31;
    const uint32_t q_bytes = (uint32_t)(2 * L::NBLK * p.G * p.tq * 128);
    const uint32_t kv_bytes = (uint32_t)(KV8 ? L::RAW_TILE : L::TILE);
    uint32_t kc = 0, vc = 0, qc = 0, vpc = 0;   // running ring / barrier counters
    int *counter = reinterpret_cast<int *>(p.ws) + 1;
    int next = blockIdx.x;                      // lane 0: the next item to hand out
    for (uint32_t n = 0; !*abort; ++n) {
        const int slot = n % IRING;
        if (n >= IRING && !mbar_wait(&bar.item_empty[slot], ((n / IRING) - 1) & 1, abort)) break;
        const int idx = __shfl_sync(0xffffffffu, next, 0);
        Item m;
        if (idx < n_items) m = load_item<MODE>(p, idx);
        else m.b = -1;                          // end of the work
        if (lane == 0) {
            bar.ring[slot] = m;
            mbar_arrive(&bar.item_full[slot]);
            // draw the following item now; the index is read one item later
            if (idx < n_items) next = (int)gridDim.x + atomicAdd(counter, 1);
        }
        if (idx >= n_items) break;
        if (m.nkt == 0) continue;
        // both Q tiles, once per item, after the previous item's BMM1s
        if (qc > 0 && !mbar_wait(bar.q_empty, (qc - 1) & 1, abort)) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar.q_full, q_bytes);
            for (int a = 0; a < 2; ++a) {
                // (debug checks) a tile with valid rows starts inside Q; a
                // tile past the item's tokens is loaded knowingly and unused
                const int tok = m.i0 + a * p.tq;
                const bool inside = tok >= m.ntok + m.i0 ||
                    dbg_ok(tok >= 0 && (p.q_packed ? m.s.q_off + tok < p.q_seq
                                                   : tok < p.q_seq && m.b < p.B) &&
                           (m.g + 1) * p.G <= p.Hq, p.status);
                for (int blk = 0; blk < L::NBLK; ++blk) {
                    if (inside)
                        tma_q(p, &tm.q, m, a, sm + L::Q_OFF + a * L::TILE + blk * L::BLK,
                              bar.q_full, blk * 64);
                    else
                        mbar_complete_tx(bar.q_full, q_bytes / (2 * L::NBLK));
                }
            }
        }
        ++qc;
        for (int t = 0; t < m.ntiles && !*abort; ++t) {
            const int j0 = key_tile<MODE>(m, t) * BN;
            const int ks = kc % L::KST;
            if (kc >= L::KST && !mbar_wait(&bar.k_empty[ks], ((kc / L::KST) - 1) & 1, abort)) break;
            if (KV8)   // bytes for the converter warps
                load_kv_tile<D, true, PAGED>(p, &tm.k, m, 0, j0, sm + L::raw_k(ks), &bar.kraw_full[ks],
                                      kv_bytes);
            else
                load_kv_tile<D, false, PAGED>(p, &tm.k, m, 0, j0, sm + L::K_OFF + ks * L::TILE,
                                       &bar.k_full[ks], kv_bytes);
            ++kc;
            if (!is_pv<MODE>(m, t)) continue;
            const int vs = vc % L::VST;
            if (vc >= L::VST && !mbar_wait(&bar.v_empty[vs], ((vc / L::VST) - 1) & 1, abort)) break;
            uint8_t *vdst = sm + L::V_OFF + vs * L::TILE;
            const int rem = m.s.kv_len - j0;
            if (KV8) {
                // the converter warps zero the rows past the sequence end
                load_kv_tile<D, true, PAGED>(p, &tm.v, m, 1, j0, sm + L::raw_v(vs), &bar.vraw_full[vs],
                                      kv_bytes);
            } else if (rem >= BN) {
                load_kv_tile<D, false, PAGED>(p, &tm.v, m, 1, j0, vdst, &bar.v_full[vs], kv_bytes);
            } else {
                // the tile runs past the sequence end: land it, clear the
                // rows past the end, then publish it
                load_kv_tile<D, false, PAGED>(p, &tm.v, m, 1, j0, vdst, bar.v_part, kv_bytes);
                const bool landed = mbar_wait(bar.v_part, vpc & 1, abort);
                ++vpc;
                if (!landed) break;
                zero_v_rows<D>(vdst, rem, lane);
                if (lane == 0) mbar_arrive(&bar.v_full[vs]);
            }
            ++vc;
        }
    }
    // Before the CTA exits, let every copy this warp started land.
    uint64_t *k_land = KV8 ? bar.kraw_full : bar.k_full;
    uint64_t *v_land = KV8 ? bar.vraw_full : bar.v_full;
    for (uint32_t c = kc > L::KST ? kc - L::KST : 0; c < kc; ++c)
        mbar_wait_drain(&k_land[c % L::KST], (c / L::KST) & 1);
    for (uint32_t c = vc > L::VST ? vc - L::VST : 0; c < vc; ++c)
        mbar_wait_drain(&v_land[c % L::VST], (c / L::VST) & 1);
    if (qc > 0) mbar_wait_drain(bar.q_full, (qc - 1) & 1);
    if (vpc > 0) mbar_wait_drain(bar.v_part, (vpc - 1) & 1);
}

// ------------------------------------------------------------------ converter (KV8)
// Expands a byte tile of E4M3 codes (128 rows x D bytes) into the 16-bit tile
// a TMA load of 16-bit values would have produced: NBLK blocks of 128 rows x
// 128 bytes, 16-byte chunks swizzled with the row's low three bits.  Lane l
// of converter warp w takes, per step, row r = r0 + l / (D/16) and its
// 16-byte chunk c = l % (D/16) (codes 16c .. 16c+15, exactly converted to
// f16 or bf16), which land in block c / 4 as the logical chunks 2(c%4) and
// 2(c%4)+1 of the row.  (D = 128: the four rows of a step are permuted
// among the quarter warps, row dr(l) = (q & 2) + ((q ^ (c >> 2)) & 1) with
// q = l / 8, so that the 8 lanes the shared memory serves together read 128
// distinct bytes and write to blocks 0 and 1 of two rows of opposite
// swizzle parity: no bank conflicts either way.)  Rows from `zero_from` on
// are written as zeros.  The
// warp reads the bytes of EB steps' rows before it writes any of them (the
// loads overlap instead of each waiting out the one before), so the
// expansion may overwrite the byte tile in place (D = 128: each 16-bit row
// of the second block covers exactly the byte row of the same index, and
// each row belongs to one warp and one batch).
template <int D, bool BF16>
__device__ __forceinline__ void expand_tile(const uint8_t *raw, uint8_t *dst, int zero_from,
                                            int w) {
    constexpr int CPR = D / 16;             // 16-byte chunks per byte row
    constexpr int RPS = 32 / CPR;           // rows per warp step
    constexpr int STEPS = BN / (2 * RPS);   // steps of one warp (two warps per tile)
    constexpr int EB = D == 128 ? 8 : 4;    // steps per batch of loads
    static_assert(STEPS % EB == 0, "whole batches");
    const int lane = threadIdx.x & 31;
    const int c = lane % CPR;
    const int l0 = 2 * (c % 4);
    const int q = lane / CPR;
    const int dr = D == 128 ? (q & 2) + ((q ^ (c >> 2)) & 1) : q;   // row within the step
#pragma unroll 1
    for (int s0 = 0; s0 < STEPS; s0 += EB) {
        uint4 b[EB];
#pragma unroll
        for (int i = 0; i < EB; ++i) {
            const int r = (w + 2 * (s0 + i)) * RPS + dr;
            b[i] = *reinterpret_cast<const uint4 *>(raw + r * D + c * 16);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < EB; ++i) {
            const int r = (w + 2 * (s0 + i)) * RPS + dr;
            uint32_t h[8];
            e4m3x4_to_x2<BF16>(b[i].x, h[0], h[1]);
            e4m3x4_to_x2<BF16>(b[i].y, h[2], h[3]);
            e4m3x4_to_x2<BF16>(b[i].z, h[4], h[5]);
            e4m3x4_to_x2<BF16>(b[i].w, h[6], h[7]);
            if (r >= zero_from) {
#pragma unroll
                for (int k = 0; k < 8; ++k) h[k] = 0u;
            }
            uint8_t *row = dst + (c / 4) * PfLayout<D>::BLK + r * 128;
            *reinterpret_cast<uint4 *>(row + ((l0 ^ (r & 7)) * 16)) =
                make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(row + (((l0 + 1) ^ (r & 7)) * 16)) =
                make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

// Largest finite |x| of a converter warp's rows (64 of 128) of a bf16 Q tile,
// as bf16 magnitude bits (non-finite values, such as NaN padding rows, are
// left out).  Lane l reads 16-byte chunks l, l + 32, ... of the rows.  A
// first pass takes the largest magnitude bits of every element two at a
// time (max.u16x2); only when that finds a non-finite value does a second
// pass compare element by element and leave those out.
template <int D>
__device__ __forceinline__ uint32_t q_tile_max(const uint8_t *tile, int w) {
    constexpr int CHUNKS = 64 * D * 2 / 16;    // 16-byte chunks in 64 rows
    const int lane = threadIdx.x & 31;
    auto chunk = [&](int c) {
        // row r = 64 w + c / (D / 8) lies in 64-column block (c % (D/8)) / 8
        const int r = 64 * w + c / (D / 8), cc = c % (D / 8);
        return *reinterpret_cast<const uint4 *>(tile + (cc / 8) * PfLayout<D>::BLK + r * 128 +
                                                (cc % 8) * 16);
    };
    uint32_t acc = 0;
#pragma unroll 4
    for (int c = lane; c < CHUNKS; c += 32) {
        const uint4 v = chunk(c);
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm("max.u16x2 %0, %0, %1;" : "+r"(acc) : "r"(ws[k] & 0x7fff7fffu));
    }
    uint32_t mx = max(acc & 0xffffu, acc >> 16);
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx < 0x7f80u) return mx;              // every element finite
    mx = 0;
    for (int c = lane; c < CHUNKS; c += 32) {
        const uint4 v = chunk(c);
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const uint32_t m16 = (ws[k] >> (16 * hlf)) & 0x7fffu;
                if ((m16 & 0x7f80u) != 0x7f80u && m16 > mx) mx = m16;
            }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    return mx;
}

// Power-of-two exponent s that puts the largest |q| (bf16 bits m16) in
// [2^14, 2^15): every component above 2^-28 of it is then an exact f16.
__device__ __forceinline__ int q_shift(uint32_t m16) {
    if (m16 == 0) return 0;
    const int e = (int)(m16 >> 7) - 127;       // floor(log2) of a normal bf16 (subnormal: -127)
    const int sft = 14 - e;
    return sft > 126 ? 126 : sft;
}

// In place: the converter warp's rows of a bf16 Q tile become f16 values of
// q * 2^s (elementwise on 16-byte chunks, so the 128-byte swizzle is kept).
// Eight chunks are read before any is written back, so the loads overlap.
template <int D>
__device__ __forceinline__ void q_tile_to_f16(uint8_t *tile, int w, float scale) {
    constexpr int CHUNKS = 64 * D * 2 / 16;
    constexpr int QB = 8;
    static_assert(CHUNKS % (32 * QB) == 0, "whole batches");
    const int lane = threadIdx.x & 31;
    uint64_t sc2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(sc2) : "f"(scale));
#pragma unroll 1
    for (int c0 = lane; c0 < CHUNKS; c0 += 32 * QB) {
        uint4 *ptr[QB];
        uint4 v[QB];
#pragma unroll
        for (int i = 0; i < QB; ++i) {
            const int c = c0 + 32 * i;
            const int r = 64 * w + c / (D / 8), cc = c % (D / 8);
            ptr[i] = reinterpret_cast<uint4 *>(tile + (cc / 8) * PfLayout<D>::BLK + r * 128 +
                                               (cc % 8) * 16);
            v[i] = *ptr[i];
        }
#pragma unroll
        for (int i = 0; i < QB; ++i) {
            uint32_t *ws = reinterpret_cast<uint32_t *>(&v[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // both halves as f32, times 2^s in one packed multiply
                uint64_t x;
                asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(ws[k] << 16), "r"(ws[k] & 0xffff0000u));
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(sc2));
                float lo, hi;
                asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
                __half2 hh = __floats2half2_rn(lo, hi);
                ws[k] = *reinterpret_cast<uint32_t *>(&hh);
            }
            *ptr[i] = v[i];
        }
    }
}

// Converter warp w (0 or 1) of an FP8 KV cache: follows the producer's K and
// V tiles item by item, expands each landed byte tile (each warp half the
// rows) into OPB (bf16) or f16 values and publishes it to the tensor core
// (k_full / v_full take one arrival per converter warp).  V rows past the
// sequence end become zeros (their codes may be NaN, and 0 * NaN would reach
// O).  QCONV (softmax with bf16 queries): the tensor core then multiplies in
// f16, so once per item the warps also turn both bf16 Q tiles into f16 in
// place, each scaled by a power of two 2^s chosen from the tile's largest
// finite |q|; 2^-s goes to shared memory for the softmax's score scale, and
// q_conv (one arrival per converter warp) publishes the tiles.
template <int D, bool OPB, bool QCONV>
__device__ __forceinline__ void convert_role(const AttnParams &p, uint8_t *sm, const PfBars &bar,
                                             volatile int *abort, int w) {
    using L = PfLayout<D, true>;
    const int lane = threadIdx.x & 31;
    float *qf = reinterpret_cast<float *>(sm + L::MISC_OFF + 16);
    uint32_t *qmax = reinterpret_cast<uint32_t *>(sm + L::MISC_OFF + 24);   // [warp][tile]
    uint32_t kc = 0, vc = 0, qc = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
        Item m;
        if (!next_item(bar, n, abort, true, m)) break;
        if (QCONV && m.nkt > 0) {
            if (!mbar_wait(bar.q_full, qc & 1, abort)) break;
            ++qc;
            for (int a = 0; a < 2; ++a) {
                const uint32_t mx = q_tile_max<D>(sm + L::Q_OFF + a * L::TILE, w);
                if (lane == 0) qmax[w * 2 + a] = mx;
            }
            asm volatile("bar.sync 7, 64;" ::: "memory");   // both converter warps
            for (int a = 0; a < 2; ++a) {
                const int sft = q_shift(max(qmax[a], qmax[2 + a]));
                q_tile_to_f16<D>(sm + L::Q_OFF + a * L::TILE, w, ldexpf(1.f, sft));
                if (w == 0 && lane == 0) qf[a] = ldexpf(1.f, -sft);
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 7, 64;" ::: "memory");   // the maxima are read; Q is written
            if (lane == 0) mbar_arrive(bar.q_conv);
        }
        for (int t = 0; t < m.ntiles; ++t) {
            const int ks = kc % L::KST;
            if (!mbar_wait(&bar.kraw_full[ks], (kc / L::KST) & 1, abort)) { ok = false; break; }
            expand_tile<D, OPB>(sm + L::raw_k(ks), sm + L::K_OFF + ks * L::TILE, BN, w);
            fence_proxy_async_smem();   // the tensor core reads what the generic proxy wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.k_full[ks]);
            ++kc;
            const int vs = vc % L::VST;
            if (!mbar_wait(&bar.vraw_full[vs], (vc / L::VST) & 1, abort)) { ok = false; break; }
            expand_tile<D, OPB>(sm + L::raw_v(vs), sm + L::V_OFF + vs * L::TILE,
                                m.s.kv_len - t * BN, w);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.v_full[vs]);
            ++vc;
        }
    }
}

// ------------------------------------------------------------------ MMA issuer
// One warp issues every tcgen05.mma, in the order
//   S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) PV1(1) S1(2) | ...
// The whole warp runs this code, converged, and one elected lane issues
// each MMA and commit: issuing from a single diverged lane instead costs
// about a third more time per MMA, and more again while the softmax warps
// sharing this warp's scheduler are busy.  Every wait result is taken from
// lane 0 so that all branches stay warp-uniform.  The hand-over from one
// GEMM to the next is kept short: descriptors and TMEM addresses are plain
// additions of constants, and the barriers the next step starts with (P_0
// and the V tile) are tested before the last MMA of S_1, while the queued
// MMAs still keep the pipe busy.
// OPB: the products' operand type is bf16 (else f16).  QCONV: the Q tiles
// are ready when the converter warps have turned them into f16 (q_conv).
template <int D, int MODE, bool OPB, bool QCONV>
__device__ __forceinline__ void mma_role(const AttnParams &p, uint8_t *sm, const PfBars &bar,
                         volatile int *abort, uint32_t tmem) {
    using L = PfLayout<D>;
    constexpr uint32_t ID_S = idesc_f16(OPB ? 1 : 0, 128, BN, 0, 0);   // Q K-major, K K-major
    constexpr uint32_t ID_O = idesc_f16(OPB ? 1 : 0, 128, D, 0, 1);    // P from TMEM, V MN-major
    constexpr int NS = D / 16;      // MMAs of one BMM1 (16 of the head dimension each)
    constexpr int NO = BN / 16;     // MMAs of one BMM2 (16 keys each)
    // A descriptor's start-address field holds addr >> 4, so a byte offset
    // o moves a descriptor by o >> 4 (every address stays below 256 KB).
    constexpr uint64_t TILE16 = L::TILE >> 4;
    const uint64_t dq0 = sdesc(smem_u32(sm + L::Q_OFF), 16, 1024);
    const uint64_t dk0 = sdesc(smem_u32(sm + L::K_OFF), 16, 1024);
    const uint64_t dv0 = sdesc(smem_u32(sm + L::V_OFF), L::BLK, 1024);
    uint32_t kc = 0, vc = 0, qc = 0, tc = 0;   // ring counters; tc: BMM1 steps per tile, running
    bool ok = true;
    auto wwait = [&](uint64_t *b, uint32_t parity, volatile int *ab) -> bool {
        return __shfl_sync(0xffffffffu, mbar_wait(b, parity, ab) ? 1 : 0, 0) != 0;
    };
    auto wtest = [&](uint32_t b, uint32_t parity) -> bool {
        return __shfl_sync(0xffffffffu, mbar_test(b, parity) ? 1 : 0, 0) != 0;
    };

    // k-step kk of S_a = Q_a K^T: 16 columns of the 128-byte swizzled rows,
    // four k-steps per 64-column block
    auto s_mma = [&](int a, uint64_t dk, int kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * L::BLK + (kk & 3) * 32) >> 4);
        mma_ss_w(tmem + S_COL0 + a * 128, dq0 + a * TILE16 + off, dk + off, ID_S, kk > 0 ? 1u : 0u);
    };
    // k-step kk of O_a (+)= P_a V: 16 keys, i.e. 8 packed TMEM columns of
    // P_a and 16 rows (2 KB) of the MN-major V tile
    auto o_mma = [&](int a, uint64_t dv, int kk, bool acc) {
        mma_ts_w(tmem + O_COL0 + a * D, tmem + S_COL0 + a * 128 + kk * 8,
               dv + (uint64_t)((kk * 2048) >> 4), ID_O, acc ? 1u : 0u);
    };

    for (uint32_t n = 0; ok; ++n) {
        Item m;
        if (!next_item(bar, n, abort, true, m)) break;
        if (m.nkt == 0) continue;
        if (!wwait(QCONV ? bar.q_conv : bar.q_full, qc & 1, abort)) break;
        ++qc;
        // S0(0), S1(0)
        int ks = kc % L::KST;
        if (!wwait(&bar.k_full[ks], (kc / L::KST) & 1, abort)) break;
        tc_fence_after();
        {
            const uint64_t dk = dk0 + ks * TILE16;
#pragma unroll
            for (int kk = 0; kk < NS; ++kk) s_mma(0, dk, kk);
            mma_commit_w(&bar.s_full[0]);
#pragma unroll
            for (int kk = 0; kk < NS; ++kk) s_mma(1, dk, kk);
            mma_commit_w(&bar.s_full[1]);
            mma_commit_w(&bar.k_empty[ks]);
            ++kc;
            if (m.ntiles == 1) mma_commit_w(bar.q_empty);
        }
        int u = 0;                                // BMM2 steps of this item
        bool p0_ready = false, v_ready = false;   // found complete ahead of time
        for (int t = 0; t < m.ntiles; ++t) {
            const bool pv = is_pv<MODE>(m, t);
            const bool more = t + 1 < m.ntiles;
            const int vs = vc % L::VST;
            const uint64_t dv = dv0 + vs * TILE16;
            if (pv && !v_ready && !wwait(&bar.v_full[vs], (vc / L::VST) & 1, abort)) { ok = false; break; }
            // P_0(t) ready (or, for a statistics step, S_0(t) consumed)
            if (!p0_ready && !wwait(&bar.p_full[0], tc & 1, abort)) { ok = false; break; }
            tc_fence_after();
            if (pv) {                             // PV0(t)
#pragma unroll
                for (int kk = 0; kk < NO; ++kk) o_mma(0, dv, kk, u > 0 || kk > 0);
                mma_commit_w(&bar.o_done[0]);
            }
            ks = kc % L::KST;
            const uint64_t dk = dk0 + ks * TILE16;
            if (more) {                           // S0(t+1)
                if (!wwait(&bar.k_full[ks], (kc / L::KST) & 1, abort)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < NS; ++kk) s_mma(0, dk, kk);
                mma_commit_w(&bar.s_full[0]);
            }
            if (!wwait(&bar.p_full[1], tc & 1, abort)) { ok = false; break; }
            tc_fence_after();
            if (pv) {                             // PV1(t); V(t) is free once it completes
#pragma unroll
                for (int kk = 0; kk < NO; ++kk) o_mma(1, dv, kk, u > 0 || kk > 0);
                mma_commit_w(&bar.o_done[1]);
                mma_commit_w(&bar.v_empty[vs]);
                ++vc;
                ++u;
            }
            ++tc;
            p0_ready = v_ready = false;
            if (more) {                           // S1(t+1)
#pragma unroll
                for (int kk = 0; kk < NS; ++kk) {
                    if (kk == NS - 1) {
                        // neither barrier can run a phase past these tests:
                        // their next phases need S_0(t+2) and the release
                        // of V(t+1), both still to come from this thread
                        p0_ready = wtest(smem_u32(&bar.p_full[0]), tc & 1);
                        v_ready = !is_pv<MODE>(m, t + 1) ||
                                  wtest(smem_u32(&bar.v_full[vc % L::VST]), (vc / L::VST) & 1);
                    }
                    s_mma(1, dk, kk);
                }
                mma_commit_w(&bar.s_full[1]);
                mma_commit_w(&bar.k_empty[ks]);
                ++kc;
                if (t + 1 == m.ntiles - 1) mma_commit_w(bar.q_empty);
            }
        }
    }
}

// ------------------------------------------------------------------ softmax
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Mask forms handled on the partial-tile path.
enum MaskKind { MK_BITS = 0, MK_ADD_F16 = 1, MK_ADD_BF16 = 2, MK_ADD_F32 = 3 };

template <typename T>
__device__ __forceinline__ float ld_as_float(const void *base, long long e) {
    if constexpr (sizeof(T) == 4) return static_cast<const float *>(base)[e];
    else if constexpr (std::is_same<T, __half>::value)
        return __half2float(static_cast<const __half *>(base)[e]);
    else return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[e]);
}

// Marker of an excluded pair in 'none' scores: a NaN whose bits no
// arithmetic produces (the GPU's arithmetic NaN is 0x7fffffff), so that an
// allowed pair whose additive mask value is -inf keeps its -inf score, as
// the plain formula does, while excluded pairs contribute 0.
constexpr uint32_t NONE_EXCLUDED = 0xffc0dead;

// Chunk c (keys j0 + 32c .. j0 + 32c + 31) of a partial tile, scaled and
// masked in place.  Key kk = 32c + k is allowed when kk <= rem (causal and
// length limits) and its bit is set: bit (kk >> 2) of word (kk & 3).
// Writes log2-domain scores (softmax), where an excluded pair is -inf, or
// natural-unit scores ('none'), where it is NONE_EXCLUDED.
// sc: the score scale (log2 units for softmax; times s_k for an FP8 cache).
template <bool LOG2, int MK>
__device__ __forceinline__ void mask_chunk(const AttnParams &p, float (&v)[32], int c, int rem,
                                           const uint32_t (&bits)[4], long long mrow, int j0,
                                           float sc) {
    const bool keyb = p.md[3] == 1;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const int kk = c * 32 + k;
        bool ok = kk <= rem;
        float val = v[k] * sc;
        if constexpr (MK == MK_BITS) {
            ok = ok && ((bits[k & 3] >> (8 * c + (k >> 2))) & 1u);
        } else {
            if (ok) {
                const long long e = keyb ? mrow : mrow + j0 + kk;
                ok = dbg_ok(e >= 0 && e < mask_elems(p), p.status);
            }
            if (ok) {
                const long long e = keyb ? mrow : mrow + j0 + kk;
                float add;
                if constexpr (MK == MK_ADD_F16) add = ld_as_float<__half>(p.mask, e);
                else if constexpr (MK == MK_ADD_BF16) add = ld_as_float<__nv_bfloat16>(p.mask, e);
                else add = ld_as_float<float>(p.mask, e);
                val += LOG2 ? add * LOG2E : add;
            }
        }
        v[k] = ok ? val : (LOG2 ? -INFINITY : __uint_as_float(NONE_EXCLUDED));
    }
}

template <bool LOG2>
__device__ __forceinline__ void mask_chunk_any(const AttnParams &p, int mk, float (&v)[32], int c,
                                               int rem, const uint32_t (&bits)[4],
                                               long long mrow, int j0, float sc) {
    switch (mk) {
    case MK_ADD_F16: mask_chunk<LOG2, MK_ADD_F16>(p, v, c, rem, bits, mrow, j0, sc); break;
    case MK_ADD_BF16: mask_chunk<LOG2, MK_ADD_BF16>(p, v, c, rem, bits, mrow, j0, sc); break;
    case MK_ADD_F32: mask_chunk<LOG2, MK_ADD_F32>(p, v, c, rem, bits, mrow, j0, sc); break;
    default: mask_chunk<LOG2, MK_BITS>(p, v, c, rem, bits, mrow, j0, sc); break;
    }
}

__device__ __forceinline__ float chunk_max(const float (&v)[32]) {
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        m0 = fmax3(m0, v[k], v[k + 1]);
        m1 = fmax3(m1, v[k + 2], v[k + 3]);
        m2 = fmax3(m2, v[k + 4], v[k + 5]);
        m3 = fmax3(m3, v[k + 6], v[k + 7]);
    }
    return fmax3(fmaxf(m0, m1), m2, m3);
}

__device__ __forceinline__ void as_float(const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

// Bitmap of allowed keys j0 .. j0+127 for a bool mask: bit (c >> 2) of
// word (c & 3) is key c.  When the mask does not depend on the query row
// (it broadcasts over heads and query positions) the warp builds it
// together with four ballots; otherwise each thread reads its own row.
__device__ __forceinline__ void mask_bits(const AttnParams &p, bool row_indep, long long mrow,
                                          int j0, int kv_len, bool row_ok, uint32_t (&bits)[4]) {
    const uint8_t *mk = static_cast<const uint8_t *>(p.mask);
    const bool keyb = p.md[3] == 1;
    if (row_indep) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = j0 + lane * 4 + k;
            const long long e = keyb ? mrow : mrow + j;
            const bool ok = j < kv_len && dbg_ok(e >= 0 && e < mask_elems(p), p.status) &&
                            mk[e] != 0;
            bits[k] = __ballot_sync(0xffffffffu, ok);
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) bits[k] = 0;
    if (!row_ok) return;
    const uint8_t *src = mk + (keyb ? mrow : mrow + j0);
    if (!keyb && j0 + BN <= kv_len && j0 + BN <= p.md[3] &&
        (reinterpret_cast<uintptr_t>(src) & 7) == 0 &&
        dbg_ok(mrow + j0 >= 0 && mrow + j0 + BN <= mask_elems(p), p.status)) {
        // the tile lies inside the mask row and the sequence: 16 loads of 8
        // key bytes each; key 8q + e lands in bits[e & 3], bit 2q + (e >> 2)
#pragma unroll
        for (int q = 0; q < BN / 8; ++q) {
            const uint2 w = *reinterpret_cast<const uint2 *>(src + 8 * q);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t byte = ((e < 4 ? w.x : w.y) >> (8 * (e & 3))) & 0xffu;
                if (byte) bits[e & 3] |= 1u << (2 * q + (e >> 2));
            }
        }
        return;
    }
#pragma unroll 1
    for (int c = 0; c < BN; ++c) {
        const int j = j0 + c;
        const long long e = keyb ? mrow : mrow + j;
        if (j < kv_len && dbg_ok(e >= 0 && e < mask_elems(p), p.status) && mk[e] != 0) {
            const uint32_t bit = 1u << (c >> 2);
            switch (c & 3) {   // a switch keeps bits[] in registers
            case 0: bits[0] |= bit; break;
            case 1: bits[1] |= bit; break;
            case 2: bits[2] |= bit; break;
            default: bits[3] |= bit; break;
            }
        }
    }
}

// Output row geometry of row r of query tile a (the same mapping as the Q
// tile): element offset of Y[token, head, 0] and whether it is written.
struct RowOut {
    long long off;
    bool ok;
};
__device__ __forceinline__ RowOut row_out(const AttnParams &p, const Item &m, int a, int r) {
    const int t = p.q_packed ? r / p.G : r % p.tq;
    const int hh = p.q_packed ? r % p.G : r / p.tq;
    const int tok = a * p.tq + t;
    const int i = m.i0 + tok;
    const int h = m.g * p.G + hh;
    RowOut o;
    o.ok = r < p.G * p.tq && tok < m.ntok;
    o.off = p.q_packed ? ((long long)(m.s.q_off + i) * p.Hq + h) * p.D
                       : (((long long)m.b * p.Hq + h) * p.q_seq + i) * p.D;
    return o;
}

// Epilogue of one row per thread: O (TMEM, fp32) * f -> 16-bit -> Y, 64
// columns at a time through the warpgroup's 16 KB staging area (row r at
// r * 128 bytes, 16-byte chunks swizzled as TMA's 128-byte swizzle does, so
// the four warps' buffers form one TMA box of the tile).
//  - tile entirely inside the sequence: one thread stores the box with TMA,
//    asynchronously; the staging is reused only after the store has read it
//    (`pending` carries that over to the next epilogue);
//  - tile running past the end of the sequence: each warp writes its own 32
//    rows, four whole 128-byte lines per instruction, skipping rows outside.
// zero: write zeros (the item has no attendable key).
template <int D, bool BF16>
__device__ __forceinline__ void store_rows(const AttnParams &p, const TensorMaps &tm,
                                           const Item &m, int a, uint32_t o_taddr, float f,
                                           bool zero, uint8_t *stg_wg, bool &pending) {
    const int lane = threadIdx.x & 31;
    const int r = threadIdx.x & 127;                  // this thread's row
    const int wr0 = r & ~31;                          // first row of this warp
    const bool whole = (a + 1) * p.tq <= m.ntok;
    uint16_t *y = static_cast<uint16_t *>(p.y);
    uint8_t *stg = stg_wg + wr0 * 128;                // this warp's 32 rows
    uint32_t v[D / 32][32];
    if (!zero) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(o_taddr + c * 32, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_regs_ready(v[c]);
    }
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
        if (pending) {   // the previous TMA store must have read the staging
            if (r == 0) bulk_wait_read();
            named_sync(1 + a, 128);
            pending = false;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = half * 64 + q * 8 + 2 * e;
                w[e] = zero ? 0u : pack2<BF16>(__uint_as_float(v[col / 32][col % 32]) * f,
                                               __uint_as_float(v[col / 32][col % 32 + 1]) * f);
            }
            *reinterpret_cast<uint4 *>(stg + lane * 128 + ((q ^ (lane & 7)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (whole) {
            fence_proxy_async_smem();
            named_sync(1 + a, 128);
            const int tok = m.i0 + a * p.tq;
            // (debug checks) the stored tile lies inside the sequence and Y
            if (r == 0 &&
                dbg_ok(tok >= 0 && tok + p.tq <= m.s.q_len && (m.g + 1) * p.G <= p.Hq &&
                       (p.q_packed ? m.s.q_off + tok + p.tq <= p.q_seq
                                   : tok + p.tq <= p.q_seq && m.b < p.B), p.status)) {
                if (p.q_packed)
                    tma_store_3d(&tm.y, stg_wg, half * 64, m.g * p.G, m.s.q_off + tok);
                else
                    tma_store_4d(&tm.y, stg_wg, half * 64, tok, m.g * p.G, m.b);
                bulk_commit();
            }
            pending = true;
        } else {
            __syncwarp();
            // four rows per instruction: lanes 8j..8j+7 write row 4k+j
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int lr = 4 * k + (lane >> 3), q = lane & 7;
                const RowOut o = row_out(p, m, a, wr0 + lr);
                const uint4 val =
                    *reinterpret_cast<const uint4 *>(stg + lr * 128 + ((q ^ (lr & 7)) * 16));
                const long long e = o.off + half * 64 + q * 8;
                if (o.ok && dbg_ok(e >= 0 && e + 8 <= q_elems(p), p.status))
                    *reinterpret_cast<uint4 *>(y + e) = val;
            }
            __syncwarp();
        }
    }
}

// Scores of a chunk past key `last` (chunk-relative) become -inf.
__device__ __forceinline__ void mask_after(uint32_t (&r)[32], int last) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (k > last) r[k] = 0xff800000u;
}

// Scores of chunk c whose key is excluded by a row-independent bool mask
// become -inf.  bits[k] bit L is key 4L + k of the tile (mask_bits, ballot).
__device__ __forceinline__ void mask_keys(uint32_t (&r)[32], const uint32_t (&bits)[4], int c) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (!((bits[i & 3] >> (8 * c + (i >> 2))) & 1u)) r[i] = 0xff800000u;
}

// Sum of 2^(s * mul - ref) over one 32-score chunk (statistics pass).
__device__ __forceinline__ void sum_chunk(const uint32_t (&r)[32], uint64_t mul2, uint64_t neg2,
                                          uint64_t &acc0, uint64_t &acc1) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float pa, pb;
        f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])), mul2, neg2),
                  pa, pb);
        pa = ex2(pa);
        pb = ex2(pb);
        if (k & 1) acc1 = fadd2(acc1, f2_pack(pa, pb));
        else acc0 = fadd2(acc0, f2_pack(pa, pb));
    }
}

// One 32-column chunk of the quantized pass: x = 2^(s * mul - ref) (with
// ref = log2 of l * s_q, x is p / s_q), rounded to the fp8 E4M3 (QK 0)
// or int8 (QK 1) grid, stored as 16-bit pairs into TMEM columns
// [16c, 16c+16) of the S buffer (every code is exact in f16 and bf16).
template <bool BF16, int QK>
__device__ __forceinline__ void p_chunk_q(const uint32_t (&r)[32], uint32_t s_addr, int c,
                                          uint64_t mul2, uint64_t neg2) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float pa, pb;
        f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])), mul2, neg2),
                  pa, pb);
        pa = ex2(pa);
        pb = ex2(pb);
        if constexpr (QK == 0) {
            uint16_t q;
            uint32_t h;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(pb), "f"(pa));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(q));
            if constexpr (BF16) {
                const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h));
                w[k] = pack2<true>(f.x, f.y);
            } else {
                w[k] = h;
            }
        } else {
            int8_round2(pa, pb);
            w[k] = pack2<BF16>(pa, pb);
        }
    }
    tmem_st16(s_addr + c * 16, w);
}

// Largest of 32 scores held as raw bits.
__device__ __forceinline__ float reg_max(const uint32_t (&r)[32]) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
    return chunk_max(v);
}

// One 32-column chunk of a full tile: p = 2^(s * mul - ref) packed to 16-bit
// pairs into TMEM columns [16c, 16c+16) of the S buffer; accumulates the
// sum of p.
template <bool BF16>
__device__ __forceinline__ void p_chunk(const uint32_t (&r)[32], uint32_t s_addr, int c,
                                        uint64_t mul2, uint64_t neg2, uint64_t &acc0,
                                        uint64_t &acc1) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float pa, pb;
        f2_unpack(ffma2(f2_pack(v[2 * k], v[2 * k + 1]), mul2, neg2), pa, pb);
        pa = ex2(pa);
        pb = ex2(pb);
        if (k & 1) acc1 = fadd2(acc1, f2_pack(pa, pb));
        else acc0 = fadd2(acc0, f2_pack(pa, pb));
        w[k] = pack2<BF16>(pa, pb);
    }
    tmem_st16(s_addr + c * 16, w);
}

// QK: the quantized op's P grid (0 fp8, 1 int8; 0 for the other modes), a
// constant of each copy of this role so that no loop carries the other
// grid's rounding.  PLAIN: softmax with no mask and a positive score scale
// (times the FP8 cache's s_k), where every tile takes the register path:
// that copy holds no general path.
template <int D, int MODE, bool BF16, bool KV8, int QK, bool PLAIN = false>
__device__ __forceinline__ void softmax_role(const AttnParams &p, const TensorMaps &tm,
                                             const PfBars &bar, volatile int *abort,
                                             int n_items, uint32_t tmem, int a, uint8_t *stg) {
    constexpr bool SOFTMAX = (MODE == MODE_SOFTMAX || MODE == MODE_SOFTMAX_Q);
    constexpr bool QUANT = (MODE == MODE_SOFTMAX_Q || MODE == MODE_NONE_Q);
    // P's type for BMM2, and whether the converter warps scale Q (FP8 cache,
    // softmax, bf16 queries: the products run in f16)
    constexpr bool OPB = BF16 && !(KV8 && MODE == MODE_SOFTMAX);
    constexpr bool QCONV = KV8 && BF16 && MODE == MODE_SOFTMAX;
    const int r = threadIdx.x & 127;                 // row = TMEM lane
    const uint32_t lane_base = (uint32_t)((r & ~31) << 16);
    const uint32_t s_addr = tmem + lane_base + S_COL0 + a * 128;
    const uint32_t o_addr = tmem + lane_base + O_COL0 + a * D;
    const int G = p.G, TQ = p.tq;
    const int t_row = p.q_packed ? r / G : r % TQ;
    const int hh = p.q_packed ? r % G : r / TQ;
    const bool in_tile = r < G * TQ;
    const float qs = QUANT ? load_qscale(p) : 1.f;
    const float inv_qs = 1.f / qs;
    // score scale; an FP8 cache folds s_k into it and s_v into the epilogue
    const float sc0 = (SOFTMAX ? p.scale_log2 : p.scale) * (KV8 ? __ldg(p.k_scale) : 1.f);
    float sc = sc0;   // per item: times 2^-s of the tile's Q scaling (QCONV)
    uint32_t qcv = 0;
    const float sv = KV8 ? __ldg(p.v_scale) : 1.f;
    const bool use_mask = !PLAIN && p.mask != nullptr;
    const bool bool_mask = use_mask && p.mask_dtype == 3;
    const bool row_indep = bool_mask && p.md[1] == 1 && p.md[2] == 1;
    const int mk = !use_mask || bool_mask ? MK_BITS
                   : p.mask_dtype == 0 ? MK_ADD_F16 : p.mask_dtype == 1 ? MK_ADD_BF16 : MK_ADD_F32;
    uint32_t tc = 0, npv = 0;                        // steps seen; BMM2s of this tile so far
    bool ok = true, pending = false;

    for (uint32_t n = 0; ok; ++n) {
        Item m;
        if (!next_item(bar, n, abort, true, m)) break;
        const int tok = a * TQ + t_row;              // token within the item
        const int i = m.i0 + tok;
        const int h = m.g * G + hh;
        const bool row_ok = in_tile && tok < m.ntok;
        if (m.nkt == 0) {                            // no attendable key: the rows are zero
            store_rows<D, BF16>(p, tm, m, a, 0, 0.f, true, stg, pending);
            continue;
        }
        if (QCONV) {   // this tile's Q scaling, once the converter warps are done
            if (!mbar_wait(bar.q_conv, qcv & 1, abort)) { ok = false; break; }
            ++qcv;
            sc = sc0 * reinterpret_cast<const volatile float *>(
                           reinterpret_cast<const uint8_t *>(bar.q_full) +
                           (PfLayout<D, KV8>::MISC_OFF - PfLayout<D, KV8>::BAR_OFF) + 16)[a];
        }
        const int lim = row_ok ? min(causal_limit(p.causal, i, m.s), m.s.kv_len - 1) : -1;
        const int lim_first = min(causal_limit(p.causal, m.i0 + a * TQ, m.s), m.s.kv_len - 1);
        const long long mrow = !use_mask ? 0
                               : row_indep ? mask_row(p, m.b, 0, 0)
                               : row_ok ? mask_row(p, m.b, h, i) : 0;
        float m_ref = -INFINITY, l = 0.f, lse2 = 0.f;
        int u = 0;
        for (int t = 0; t < m.ntiles; ++t) {
            const int j0 = key_tile<MODE>(m, t) * BN;
            // the bool mask's bits of the tile, read while S is computed
            uint32_t bits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            if (bool_mask) mask_bits(p, row_indep, mrow, j0, m.s.kv_len, row_ok, bits);
            if (!mbar_wait(&bar.s_full[a], tc & 1, abort)) { ok = false; break; }
            tc_fence_after();
            const int rem = lim - j0;
            const bool full = !use_mask && j0 + BN - 1 <= lim_first && (PLAIN || sc > 0.f);
            const bool stat = (MODE == MODE_SOFTMAX_Q) && t < m.nkt;
            // a row-independent bool mask that keeps every key of the tile
            // needs no per-score test (warp-uniform: the bits are the warp's)
            const bool mask_part =
                use_mask && (!row_indep || (bits[0] & bits[1] & bits[2] & bits[3]) != 0xffffffffu);

            // Softmax without an explicit mask (and the quantized op's
            // statistics and quantized passes, also under a bool mask that
            // depends on the key only): take the exps against the
            // running reference while the second half of the row is still
            // loading; redo the step only when some row's max grows past the
            // reference by more than the threshold.  Keys past a row's
            // causal or length limit (a prefix of the tile stays visible) and
            // keys the bool mask excludes become -inf in registers.  A row
            // without a reference yet takes the max of its first 64 visible
            // scores (none visible: all its p are 0).
            if (((MODE == MODE_SOFTMAX && !use_mask) ||
                 (MODE == MODE_SOFTMAX_Q && (!use_mask || row_indep))) && (PLAIN || sc > 0.f)) {
                const bool lim_full = j0 + BN - 1 <= lim_first;   // no causal/length limit in the tile
                const uint64_t mul2 = f2_pack(sc, sc);
                uint32_t ra[2][32], rb[2][32];
                tmem_ld32(s_addr, ra[0]);
                tmem_ld32(s_addr + 32, ra[1]);
                tmem_wait_ld();
                if (MODE == MODE_SOFTMAX_Q) {
                    tmem_regs_ready(ra[0]);
                    tmem_regs_ready(ra[1]);
                }
                tmem_ld32(s_addr + 64, rb[0]);
                tmem_ld32(s_addr + 96, rb[1]);
                if (!lim_full) {
                    mask_after(ra[0], rem);
                    mask_after(ra[1], rem - 32);
                }
                if (MODE == MODE_SOFTMAX_Q && mask_part) {
                    mask_keys(ra[0], bits, 0);
                    mask_keys(ra[1], bits, 1);
                }
                if (MODE == MODE_SOFTMAX_Q) {
                    tmem_wait_ld();
                    tmem_regs_ready(rb[0]);
                    tmem_regs_ready(rb[1]);
                    if (!lim_full) {
                        mask_after(rb[0], rem - 64);
                        mask_after(rb[1], rem - 96);
                    }
                    if (mask_part) {
                        mask_keys(rb[0], bits, 2);
                        mask_keys(rb[1], bits, 3);
                    }
                    if (stat) {
                        // pass 1: S is in registers, so the tensor core may
                        // already write the next S over it.  The row sum is
                        // taken against a running reference, as in the
                        // softmax pass: a row's first visible scores set it
                        // (their max); the tile max is needed again only
                        // when the sum shows a score above the reference by
                        // more than the threshold, and then the sum is
                        // retaken against the new max.  lse2 = ref + log2 l.
                        tc_fence_before();
                        mbar_arrive(&bar.p_full[a]);
                        auto tile_max = [&]() {
                            return fmaxf(fmaxf(reg_max(ra[0]), reg_max(ra[1])),
                                         fmaxf(reg_max(rb[0]), reg_max(rb[1])));
                        };
                        auto tile_sum = [&](float ref) {
                            const uint64_t neg2 = f2_pack(-ref, -ref);
                            uint64_t acc0 = 0, acc1 = 0;
                            sum_chunk(ra[0], mul2, neg2, acc0, acc1);
                            sum_chunk(ra[1], mul2, neg2, acc0, acc1);
                            sum_chunk(rb[0], mul2, neg2, acc0, acc1);
                            sum_chunk(rb[1], mul2, neg2, acc0, acc1);
                            float s0, s1, s2, s3;
                            f2_unpack(acc0, s0, s1);
                            f2_unpack(acc1, s2, s3);
                            return (s0 + s1) + (s2 + s3);
                        };
                        if (__any_sync(0xffffffffu, row_ok && m_ref == -INFINITY)) {
                            const float mx = tile_max() * sc;   // -inf: nothing visible yet
                            if (row_ok && m_ref == -INFINITY) m_ref = mx;
                        }
                        const bool has_ref = row_ok && m_ref != -INFINITY;
                        float ref = has_ref ? m_ref : 0.f;
                        float sum = tile_sum(ref);
                        const bool big = has_ref && !(sum <= RESCALE_SUM);
                        if (__any_sync(0xffffffffu, big)) {
                            const float mx = tile_max() * sc;
                            const bool grow = big && mx > m_ref;
                            if (grow) {
                                l *= ex2(m_ref - mx);
                                m_ref = mx;
                                ref = mx;
                            }
                            if (__any_sync(0xffffffffu, grow)) sum = tile_sum(ref);
                        }
                        if (has_ref) l += sum;
                        if (t == m.nkt - 1)
                            lse2 = (l > 0.f) ? m_ref + log2f(l) + log2f(qs) : INFINITY;
                        ++tc;
                        continue;
                    }
                    // pass 2: p / s_q = 2^(s sc - lse2), quantized (0 for an
                    // excluded key or a row with no key: lse2 is +inf there)
                    const uint64_t neg2 = f2_pack(-lse2, -lse2);
                    p_chunk_q<OPB, QK>(ra[0], s_addr, 0, mul2, neg2);
                    p_chunk_q<OPB, QK>(ra[1], s_addr, 1, mul2, neg2);
                    p_chunk_q<OPB, QK>(rb[0], s_addr, 2, mul2, neg2);
                    p_chunk_q<OPB, QK>(rb[1], s_addr, 3, mul2, neg2);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bar.p_full[a]);
                    ++u;
                    ++tc;
                    continue;
                }
                if (__any_sync(0xffffffffu, row_ok && m_ref == -INFINITY)) {
                    // first reference: the max of the first 64 scores
                    // (visible keys form a prefix here: no explicit mask)
                    const float m01 = fmaxf(reg_max(ra[0]), reg_max(ra[1])) * sc;
                    if (row_ok && m_ref == -INFINITY) m_ref = m01;
                }
                const float ref0 = (row_ok && m_ref != -INFINITY) ? m_ref : 0.f;
                uint64_t neg2 = f2_pack(-ref0, -ref0);
                uint64_t acc0 = 0, acc1 = 0;
                p_chunk<OPB>(ra[0], s_addr, 0, mul2, neg2, acc0, acc1);
                p_chunk<OPB>(ra[1], s_addr, 1, mul2, neg2, acc0, acc1);
                tmem_wait_ld();
                if (!lim_full) {
                    mask_after(rb[0], rem - 64);
                    mask_after(rb[1], rem - 96);
                }
                p_chunk<OPB>(rb[0], s_addr, 2, mul2, neg2, acc0, acc1);
                p_chunk<OPB>(rb[1], s_addr, 3, mul2, neg2, acc0, acc1);
                // No probability can pass 2^threshold while their sum stays
                // below it, so the row max is only needed (to decide on a
                // new reference) when the sum is that large.
                float alpha = 1.f, mx = -INFINITY;
                bool need = false;
                {
                    float s0, s1, s2, s3;
                    f2_unpack(acc0, s0, s1);
                    f2_unpack(acc1, s2, s3);
                    const bool big = row_ok && !((s0 + s1) + (s2 + s3) <= RESCALE_SUM);
                    if (__any_sync(0xffffffffu, big)) {
                        const float mraw = fmaxf(fmaxf(reg_max(ra[0]), reg_max(ra[1])),
                                                 fmaxf(reg_max(rb[0]), reg_max(rb[1])));
                        mx = row_ok ? mraw * sc : -INFINITY;
                        need = mx > m_ref + RESCALE_THRESHOLD;
                    }
                }
                if (__any_sync(0xffffffffu, need)) {   // rare: redo with the new reference
                    if (need) {
                        alpha = ex2(m_ref - mx);
                        l *= alpha;
                        m_ref = mx;
                    }
                    const float ref1 = row_ok ? m_ref : 0.f;
                    neg2 = f2_pack(-ref1, -ref1);
                    acc0 = acc1 = 0;
                    p_chunk<OPB>(ra[0], s_addr, 0, mul2, neg2, acc0, acc1);
                    p_chunk<OPB>(ra[1], s_addr, 1, mul2, neg2, acc0, acc1);
                    p_chunk<OPB>(rb[0], s_addr, 2, mul2, neg2, acc0, acc1);
                    p_chunk<OPB>(rb[1], s_addr, 3, mul2, neg2, acc0, acc1);
                }
                float s0, s1, s2, s3;
                f2_unpack(acc0, s0, s1);
                f2_unpack(acc1, s2, s3);
                l += (s0 + s1) + (s2 + s3);
                // O holds the earlier BMM2s, all complete: S of this step was
                // issued after them, and its completion covers them
                if (u > 0) {
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(o_addr + c * 32, o);
                            tmem_wait_ld();
                            tmem_regs_ready(o);
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                            tmem_st32(o_addr + c * 32, o);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full[a]);
                ++u;
                ++tc;
                continue;
            }

            // this thread's score row: one TMEM round trip for a full tile;
            // a partial tile is loaded and masked a chunk at a time, which
            // keeps the mask reads of one chunk from piling up registers
            float x[BN];
            if (full || mk == MK_BITS) {
                uint32_t rr[BN / 32][32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, rr[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_regs_ready(rr[c]);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[c * 32 + k] = __uint_as_float(rr[c][k]);
                if (!full)   // causal / length / bool-mask bits: no memory reads
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        mask_chunk<SOFTMAX, MK_BITS>(p, *reinterpret_cast<float(*)[32]>(&x[c * 32]),
                                                     c, rem, bits, mrow, j0, sc);
            } else {   // additive mask: scale and mask a chunk at a time
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(s_addr + c * 32, rr);
                    tmem_wait_ld();
                    tmem_regs_ready(rr);
                    float v[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(rr[k]);
                    mask_chunk_any<SOFTMAX>(p, mk, v, c, rem, bits, mrow, j0, sc);
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[c * 32 + k] = v[k];
                }
            }
            const float mul = full ? sc : 1.f;
            float mx = -INFINITY;
            if (MODE == MODE_SOFTMAX || stat) {
                float cm[BN / 32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    cm[c] = chunk_max(*reinterpret_cast<float(*)[32]>(&x[c * 32]));
                mx = fmax3(fmaxf(cm[0], cm[1]), cm[2], cm[3]);
                if (full) mx *= sc;
                if (!row_ok) mx = -INFINITY;
            }

            // the value subtracted inside exp2 (log2 domain)
            float ref = 0.f, alpha = 1.f;
            bool need = false;
            if (stat) {
                const float m_new = fmaxf(m_ref, mx);
                ref = (m_new == -INFINITY) ? 0.f : m_new;
            } else if (MODE == MODE_SOFTMAX) {
                const float m_new = fmaxf(m_ref, mx);
                if (m_new > m_ref + RESCALE_THRESHOLD) {
                    alpha = ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                    need = true;
                }
                ref = (m_ref == -INFINITY) ? 0.f : m_ref;
            } else if (MODE == MODE_SOFTMAX_Q) {
                ref = lse2;   // pass 2: p / s_q directly
            }

            // probabilities (or only the row sum, for a statistics step);
            // the P grid (QK: 0 fp8, 1 int8) is a constant of each copy of
            // the loop, so that no iteration carries the other rounding
            const uint64_t mul2 = f2_pack(mul, mul), neg2 = f2_pack(-ref, -ref);
            uint64_t acc0 = 0, acc1 = 0;
            auto probs = [&](auto qk) {
                constexpr int QG = decltype(qk)::value;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t w[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float pa = x[c * 32 + 2 * k], pb = x[c * 32 + 2 * k + 1];
                        if (SOFTMAX) {
                            f2_unpack(ffma2(f2_pack(pa, pb), mul2, neg2), pa, pb);
                            pa = ex2(pa);
                            pb = ex2(pb);
                            if (MODE == MODE_SOFTMAX || stat) {
                                if (k & 1) acc1 = fadd2(acc1, f2_pack(pa, pb));
                                else acc0 = fadd2(acc0, f2_pack(pa, pb));
                            }
                        } else {
                            pa = (__float_as_uint(pa) == NONE_EXCLUDED) ? 0.f : pa * mul;
                            pb = (__float_as_uint(pb) == NONE_EXCLUDED) ? 0.f : pb * mul;
                            if (MODE == MODE_NONE_Q) {
                                pa *= inv_qs;
                                pb *= inv_qs;
                            }
                        }
                        if (QUANT && !stat) {
                            if constexpr (QG == 0) {
                                const float2 e = e4m3_round2(pa, pb);
                                pa = e.x;
                                pb = e.y;
                            } else {
                                int8_round2(pa, pb);
                            }
                        }
                        w[k] = pack2<OPB>(pa, pb);
                    }
                    if (!stat) tmem_st16(s_addr + c * 16, w);
                }
            };
            probs(std::integral_constant<int, QK>{});
            float s0, s1, s2, s3;
            f2_unpack(acc0, s0, s1);
            f2_unpack(acc1, s2, s3);
            const float psum = (s0 + s1) + (s2 + s3);

            if (stat) {
                // pass 1 of the quantized softmax: exact row max and sum
                const float m_new = fmaxf(m_ref, mx);
                if (m_new != -INFINITY) {
                    l = l * ex2(m_ref - m_new) + psum;
                    m_ref = m_new;
                }
                if (t == m.nkt - 1)
                    lse2 = (l > 0.f) ? m_ref + log2f(l) + log2f(qs) : INFINITY;
                tc_fence_before();
                mbar_arrive(&bar.p_full[a]);
                ++tc;
                continue;
            }
            if (MODE == MODE_SOFTMAX) l += psum;
            // O holds the earlier BMM2s, all complete (S of this step follows them)
            if (u > 0) {
                if (MODE == MODE_SOFTMAX && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + c * 32, o);
                        tmem_wait_ld();
                        tmem_regs_ready(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(o_addr + c * 32, o);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full[a]);
            ++u;
            ++tc;
        }
        if (!ok) break;
        // epilogue: after the item's last BMM2.  o_done completes a phase per
        // BMM2; every earlier one had completed before the last S did, so
        // only the last can still be outstanding and its parity is awaited.
        npv += (MODE == MODE_SOFTMAX_Q) ? m.nkt : m.ntiles;
        if (!mbar_wait(&bar.o_done[a], (npv - 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        float f;
        if (MODE == MODE_SOFTMAX) f = (l > 0.f) ? sv / l : 0.f;
        else f = qs * sv;    // 'none': 1 (s_v); quantized: the Q/DQ scale
        store_rows<D, BF16>(p, tm, m, a, o_addr, f, false, stg, pending);
        tc_fence_before();
    }
    if (r == 0) bulk_wait_all();   // the last TMA stores complete before the CTA exits
}

// ------------------------------------------------------------------ kernel
// KV8: K and V are E4M3 codes (FP8 KV cache), expanded by warps 10-11.
template <int D, int MODE, bool BF16, bool KV8>
__global__ void __launch_bounds__(PF_THREADS, 1)
prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    constexpr bool QUANT_MODE = MODE == MODE_SOFTMAX_Q || MODE == MODE_NONE_Q;
    using L = PfLayout<D, KV8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PfBars bar = pf_bars<D, KV8>(sm + L::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::MISC_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::MISC_OFF + 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full, 1);
        mbar_init(bar.q_empty, 1);
        // with an FP8 cache the two converter warps publish each K and V tile
        const int pub = KV8 ? 2 : 1;
        for (int s = 0; s < L::KST; ++s) {
            mbar_init(&bar.k_full[s], pub);
            mbar_init(&bar.k_empty[s], 1);
            mbar_init(&bar.kraw_full[s], 1);
        }
        for (int s = 0; s < L::VST; ++s) {
            mbar_init(&bar.v_full[s], pub);
            mbar_init(&bar.v_empty[s], 1);
            mbar_init(&bar.vraw_full[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.s_full[s], 1);
            mbar_init(&bar.p_full[s], 128);
            mbar_init(&bar.o_done[s], 1);
        }
        mbar_init(bar.v_part, 1);
        mbar_init(bar.q_conv, 2);   // one arrival per converter warp
        for (int s = 0; s < IRING; ++s) {
            mbar_init(&bar.item_full[s], 1);
            mbar_init(&bar.item_empty[s], ITEM_CONSUMERS + (KV8 ? 2 : 0));
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 9 && lane == 0) {
        prefetch_tmap(&tm.q);
        prefetch_tmap(&tm.k);
        prefetch_tmap(&tm.v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the scheduler's work list is complete and visible
    const int n_items = *reinterpret_cast<volatile const int *>(p.ws);

    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(PF_SOFTMAX_REGS));
        uint8_t *stg = sm + L::STG_OFF + (warp >> 2) * 4 * L::STG_WARP;
        if (QUANT_MODE && p.quant != 0)
            softmax_role<D, MODE, BF16, KV8, 1>(p, tm, bar, abort, n_items, tmem, warp >> 2, stg);
        else if (MODE == MODE_SOFTMAX && !p.mask && p.scale > 0.f &&
                 (!KV8 || __ldg(p.k_scale) > 0.f))
            softmax_role<D, MODE, BF16, KV8, 0, MODE == MODE_SOFTMAX>(p, tm, bar, abort, n_items,
                                                                     tmem, warp >> 2, stg);
        else
            softmax_role<D, MODE, BF16, KV8, 0>(p, tm, bar, abort, n_items, tmem, warp >> 2, stg);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(PF_AUX_REGS));
    }
    if (warp < 8) {
    } else if (warp == 8) {
        mma_role<D, MODE, BF16 && !(KV8 && MODE == MODE_SOFTMAX), KV8 && BF16 && MODE == MODE_SOFTMAX>(
            p, sm, bar, abort, tmem);
    } else if (warp == 9) {
        if (p.paged) producer_role<D, MODE, KV8, true>(p, tm, sm, bar, abort, n_items);
        else producer_role<D, MODE, KV8, false>(p, tm, sm, bar, abort, n_items);
    } else if (KV8) {
        convert_role<D, BF16 && MODE != MODE_SOFTMAX, BF16 && MODE == MODE_SOFTMAX>(
            p, sm, bar, abort, warp - 10);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) tmem_dealloc(tmem, TMEM_COLS);
    if (threadIdx.x == 0 && *abort) set_status(p.status, 5);
}

template <int D, int MODE, bool BF16, bool KV8>
static cudaError_t launch_one(const AttnParams &p, const TensorMaps &m, int grid,
                              cudaStream_t s) {
    using L = PfLayout<D, KV8>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [] {
        // the register split needs exactly the launch allocation it was sized for
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, prefill_kernel<D, MODE, BF16, KV8>);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != PF_LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(prefill_kernel<D, MODE, BF16, KV8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    });
    if (e != cudaSuccess) return e;
    return launch_dependent(prefill_kernel<D, MODE, BF16, KV8>, grid, PF_THREADS, L::ALLOC, s, p,
                            m);
}

template <int D, bool BF16>
static cudaError_t launch_mode(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                               cudaStream_t s) {
    switch (mode) {
    case MODE_SOFTMAX: return launch_one<D, MODE_SOFTMAX, BF16, false>(p, m, grid, s);
    case MODE_NONE: return launch_one<D, MODE_NONE, BF16, false>(p, m, grid, s);
    case MODE_SOFTMAX_Q: return launch_one<D, MODE_SOFTMAX_Q, BF16, false>(p, m, grid, s);
    default: return launch_one<D, MODE_NONE_Q, BF16, false>(p, m, grid, s);
    }
}

// Launch for one element type; each type is instantiated in its own
// translation unit (prefill_f16.cu, prefill_bf16.cu).
template <bool BF16>
cudaError_t launch_prefill_typed(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                                 cudaStream_t s) {
    if (p.D == 64) return launch_mode<64, BF16>(p, m, mode, grid, s);
    return launch_mode<128, BF16>(p, m, mode, grid, s);
}

// Over an FP8 KV cache (softmax or 'none'; the quantized op has no FP8
// cache form), instantiated in prefill_kv8.cu.
template <bool BF16>
cudaError_t launch_prefill_kv8_typed(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                                     cudaStream_t s) {
    if (mode != MODE_SOFTMAX && mode != MODE_NONE) return cudaErrorInvalidValue;
    const bool sm = mode == MODE_SOFTMAX;
    if (p.D == 64)
        return sm ? launch_one<64, MODE_SOFTMAX, BF16, true>(p, m, grid, s)
                  : launch_one<64, MODE_NONE, BF16, true>(p, m, grid, s);
    return sm ? launch_one<128, MODE_SOFTMAX, BF16, true>(p, m, grid, s)
              : launch_one<128, MODE_NONE, BF16, true>(p, m, grid, s);
}

}  // namespace rga
