// decode_group.cu - split-KV attention for decode shapes with several
// 16-row chunks per (batch, KV head): tree decoding (a few draft tokens per
// sequence times the G query heads of a KV head), the AttentionPlugin's
// tree-attention decoding ("TensorRT Plugins Guide", AttentionPlugin) with
// the TRT_Attention semantics of "TensorRT Custom Operator Schemas".
//
// The per-warp decode kernel (decode.cuh) streams the keys of a (batch, KV
// head) once per 16-row chunk, on warps far apart in its stream-K line.
// Here the warps come in groups of four: a group takes a contiguous range of
// the line of all key tiles of all units (batch b, KV head g, round r), and
// warp w of the group computes chunk 4 r + w of the unit on every tile, so
// each K and V tile is loaded once, into the group's own ring, for up to 64
// query rows.  A unit with more than four chunks takes several rounds.  The
// group's warp 0 refills a stage once all four warps have released it; the
// four warps clear the V rows past a sequence's end together.  A chunk
// inside one group's range is written to Y by its warp; a chunk cut by range
// ends leaves a partial (O, m, l) in a slot of its warp, and the last of its
// warps to finish (atomic ticket) merges them in group order, as in the
// per-warp kernel (same workspace layout: tickets per (batch, KV head,
// chunk), two partial slots per warp of the grid).
#include "decode.cuh"

namespace rga {

constexpr int GRP_WARPS = 4;    // warps per group: one per chunk of a round
constexpr int GRP_GROUPS = 2;   // groups per CTA (8 warps: the register file holds 8 x 255)
constexpr int GRP_STAGES = 4;   // K + V stages of a group's ring

template <int D>
struct GrpLayout {
    static constexpr int THREADS = GRP_WARPS * GRP_GROUPS * 32;
    static constexpr int BLK = DEC_KEYS * 128;           // 32 rows x 64 columns x 2 bytes
    static constexpr int TILE = (D / 64) * BLK;          // one K or V tile
    static constexpr int STAGE = 2 * TILE;               // K + V
    static constexpr int GROUP_RING = GRP_STAGES * STAGE;
    static constexpr int RING = GRP_GROUPS * GROUP_RING;
    static constexpr int BAR_OFF = RING;                 // land[group][stage], empty[group][stage]
    static constexpr int NBAR = 2 * GRP_GROUPS * GRP_STAGES;
    static constexpr int ABORT_OFF = BAR_OFF + NBAR * 8;  // abort flag, bad-lengths flag
    static constexpr int SCR_OFF = ABORT_OFF + 64;       // prefix scratch
    static constexpr int TPRE_OFF = SCR_OFF + (THREADS + 1) * 4 + 12;
    static constexpr int PPRE_OFF = TPRE_OFF + (DEC_MAX_B + 1) * 4;
    static constexpr int BYTES = PPRE_OFF + (DEC_MAX_B + 1) * 4 + 64;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory per CTA");
};

// Batch b's chunks of 16 query rows, rounds of GRP_WARPS chunks and key tiles.
__device__ __forceinline__ void grp_batch_shape(const AttnParams &p, const SeqInfo &s, int &nrc,
                                                int &nround, int &nt) {
    dec_batch_shape<DEC_ROWS_WIDE>(p, s, nrc, nt);
    nround = (nrc + GRP_WARPS - 1) / GRP_WARPS;
}

// One lane's view of the unit being computed or loaded: (batch b, unit ui =
// g * nround + round) and the tile within it.
struct GrpCur {
    int b, ui, tile;
    int nt, nrc, nround;
    SeqInfo s;
};

template <int D, bool BF16, bool SOFTMAX, bool PAGED>
__global__ void __launch_bounds__(GrpLayout<D>::THREADS, 1)
decode_group_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    using L = GrpLayout<D>;
    constexpr int NB = 2, DR = 16, NS = GRP_STAGES, NO = D / 16, KS = D / 16;
    constexpr int DLAY = DLAY_16T;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::ABORT_OFF);
    int *flags = reinterpret_cast<int *>(sm + L::ABORT_OFF + 4);
    int *scratch = reinterpret_cast<int *>(sm + L::SCR_OFF);
    int *tpre = reinterpret_cast<int *>(sm + L::TPRE_OFF);   // key tiles before batch b
    int *ppre = reinterpret_cast<int *>(sm + L::PPRE_OFF);   // (KV head, chunk) pairs before b
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = warp / GRP_WARPS, w = warp % GRP_WARPS;   // group, chunk lane
    uint64_t *land = bars + gi * NS;
    uint64_t *empty = bars + GRP_GROUPS * NS + gi * NS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < GRP_GROUPS * NS; ++i) {
            mbar_init(&bars[i], 1);                          // land: the TMA's transactions
            mbar_init(&bars[GRP_GROUPS * NS + i], GRP_WARPS);  // empty: one arrival per warp
        }
        *abort = 0;
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += L::THREADS) {
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
        if (!ok) atomicOr(&flags[0], 1);
        int nrc = 0, nround = 0, nt = 0;
        if (ok) grp_batch_shape(p, s, nrc, nround, nt);
        tpre[b] = p.Hkv * nround * nt;
        ppre[b] = p.Hkv * nrc;
    }
    __syncthreads();
    if (flags[0]) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
        return;
    }
    dec_prefix<L::THREADS>(tpre, p.B, scratch);
    dec_prefix<L::THREADS>(ppre, p.B, scratch);
    pdl_wait();   // the tickets have been cleared (and, paged, the pages checked)
    if constexpr (PAGED) {
        const volatile int *pf = reinterpret_cast<const volatile int *>(p.ws) + WS_PAGE_FLAGS;
        const int bad = (int)threadIdx.x < dec_prep_blocks(p) ? pf[threadIdx.x] : 0;
        if (__syncthreads_or(bad)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
            return;
        }
    }

    // The line: all key tiles of all units, batch-major; cut into equal
    // contiguous ranges, one per group of the grid.
    const int T = tpre[p.B];
    const int vg = blockIdx.x * GRP_GROUPS + gi;
    const int Wn = max(1, min((int)gridDim.x * GRP_GROUPS, T));
    auto range_start = [&](int v) { return (int)((long long)v * T / Wn); };
    auto group_of = [&](int x) { return (int)(((long long)(x + 1) * Wn - 1) / T); };
    int *tickets = reinterpret_cast<int *>(p.ws + dec_tickets_off(p));
    float *part = reinterpret_cast<float *>(p.ws + dec_part_off(p));
    float2 *pml = reinterpret_cast<float2 *>(p.ws + dec_ml_off(p));

    // batches with query rows but no key tile: their rows are zero
    for (int b = blockIdx.x * (L::THREADS / 32) + warp; b < p.B; b += gridDim.x * (L::THREADS / 32)) {
        const SeqInfo s = seq_info(p, b);
        int nrc, nround, nt;
        grp_batch_shape(p, s, nrc, nround, nt);
        if (nrc == 0 || nt > 0) continue;
        const int rows = s.q_len * p.G;
        for (int r = lane; r < p.Hkv * rows; r += 32) {
            const DecRow R = dec_row(p, s, b, r / rows, r % rows, rows, 0);
            if (!dbg_ok(R.qoff >= 0 && R.qoff + D <= q_elems(p), p.status)) continue;
            uint4 *y = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff);
            for (int c = 0; c < D / 8; ++c) y[c] = make_uint4(0, 0, 0, 0);
        }
    }

    uint8_t *ring = sm + gi * L::GROUP_RING;
    const uint32_t ring_u32 = smem_u32(ring);
    const int t_begin = vg < Wn ? range_start(vg) : T, t_end = vg < Wn ? range_start(vg + 1) : T;

    auto locate = [&](int t, GrpCur &c) {
        int lo = 0, hi = p.B;   // tpre[lo] <= t < tpre[lo + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tpre[mid] <= t) lo = mid; else hi = mid;
        }
        c.b = lo;
        c.s = seq_info(p, lo);
        grp_batch_shape(p, c.s, c.nrc, c.nround, c.nt);
        const int r = t - tpre[lo];
        c.ui = r / c.nt;
        c.tile = r % c.nt;
    };
    auto advance = [&](GrpCur &c) {   // the next tile of the line
        if (++c.tile < c.nt) return;
        c.tile = 0;
        if (++c.ui < p.Hkv * c.nround) return;
        int b = c.b + 1;
        while (b < p.B && tpre[b + 1] == tpre[b]) ++b;   // batches without tiles
        if (b >= p.B) return;                              // past the end: never used
        c.b = b;
        c.ui = 0;
        c.s = seq_info(p, b);
        grp_batch_shape(p, c.s, c.nrc, c.nround, c.nt);
    };
    // the group's warp 0 issues tile loads; lane 0 reads the pages
    auto issue = [&](const GrpCur &c, uint32_t n) {
        if (lane == 0) {
            int pk = 0, pv = 0;
            if constexpr (PAGED) {
                const int32_t *pt = p.page_table + (size_t)c.b * 2 * p.max_pages;
                const int pg = c.tile * DEC_KEYS / p.page_size;
                pk = __ldg(pt + pg);
                pv = __ldg(pt + p.max_pages + pg);
            }
            fence_proxy_async_smem();   // the stage's previous tile was read by ldmatrix
            dec_tma<false, PAGED>(p, tm, c.s, c.b, c.ui / c.nround, c.tile * DEC_KEYS,
                                  ring + (n % NS) * L::STAGE, &land[n % NS], D, pk, pv);
        }
    };

    const float sc = (SOFTMAX ? p.scale_log2 : p.scale);
    bool ok = true;
    uint32_t consumed = 0, issued = 0;
    if (t_begin < t_end) {
        GrpCur lc, cc;
        locate(t_begin, lc);
        cc = lc;
        if (w == 0)
            for (int t = t_begin; t < t_end && t < t_begin + NS; ++t) {
                issue(lc, issued);
                ++issued;
                advance(lc);
            }
        DecRow rr[NB][2];
        uint32_t qa[NB][KS][2];
        float o[NB][NO][4];
        float m_r[NB][2], l_r[NB][2];
        int seg0 = t_begin;   // first tile of the current unit in this range
        int kv_hi = 0, rows = 0, chunk = 0;
        bool active = false;  // this warp has a chunk of the current unit
        auto start_unit = [&]() {
            const int g = cc.ui / cc.nround, round = cc.ui % cc.nround;
            chunk = round * GRP_WARPS + w;
            active = chunk < cc.nrc;
            rows = cc.s.q_len * p.G;
            kv_hi = key_extent(p.causal, cc.s.q_len - 1, cc.s);
            const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int r0 = chunk * DR + 8 * nb;
                rr[nb][0] = dec_row(p, cc.s, cc.b, g, r0 + 2 * (lane & 3), rows, kv_hi);
                rr[nb][1] = dec_row(p, cc.s, cc.b, g, r0 + 2 * (lane & 3) + 1, rows, kv_hi);
                DecRow rq = dec_row(p, cc.s, cc.b, g, r0 + (lane >> 2), rows, kv_hi);
                rq.valid = rq.valid && dbg_ok(rq.qoff >= 0 && rq.qoff + D <= q_elems(p), p.status);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qa[nb][ks][0] = rq.valid ? q32[(rq.qoff >> 1) + 8 * ks + (lane & 3)] : 0u;
                    qa[nb][ks][1] = rq.valid ? q32[(rq.qoff >> 1) + 8 * ks + 4 + (lane & 3)] : 0u;
                }
#pragma unroll
                for (int n = 0; n < NO; ++n) o[nb][n][0] = o[nb][n][1] = o[nb][n][2] = o[nb][n][3] = 0.f;
                m_r[nb][0] = m_r[nb][1] = -INFINITY;
                l_r[nb][0] = l_r[nb][1] = 0.f;
            }
        };
        start_unit();

        for (int t = t_begin; t < t_end; ++t) {
            const uint32_t n = consumed;
            const int st = n % NS;
            if (!mbar_wait(&land[st], (n / NS) & 1, abort)) { ok = false; break; }
            ++consumed;
            const int j0 = cc.tile * DEC_KEYS;
            const uint32_t kb = ring_u32 + st * L::STAGE, vb = kb + L::TILE;
            const int rem = cc.s.kv_len - j0;
            if (rem < DEC_KEYS) {
                // V rows past the sequence end may hold NaN: the group's four
                // warps zero them together, then meet (same tile for all four)
                uint8_t *vp = ring + st * L::STAGE + L::TILE;
                constexpr int CPR = D / 8;   // 16-byte chunks per row
                for (int idx = w * 32 + lane; idx < DEC_KEYS * CPR; idx += GRP_WARPS * 32) {
                    const int row = idx / CPR, ch = idx % CPR;
                    if (row >= rem)
                        *reinterpret_cast<uint4 *>(vp + swz(row, ch, L::BLK)) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("bar.sync %0, %1;" :: "r"(1 + gi), "r"(GRP_WARPS * 32) : "memory");
            }
            if (active) dec_tile16t<D, BF16, SOFTMAX, NB>(p, rr, qa, kb, vb, j0, o, m_r, l_r, sc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (w == 0 && issued < (uint32_t)(t_end - t_begin)) {
                // refill this stage once the group's four warps have released it
                if (!mbar_wait(&empty[st], (n / NS) & 1, abort)) { ok = false; break; }
                issue(lc, issued);
                ++issued;
                advance(lc);
            }
            const bool unit_end = cc.tile + 1 == cc.nt;
            if (active && (unit_end || t + 1 == t_end)) {
                // this range's share of the chunk is done (the lanes sharing a
                // row differ in lane / 4)
                if (SOFTMAX)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int m = 4; m < 32; m <<= 1)
                                l_r[nb][r] += __shfl_xor_sync(0xffffffffu, l_r[nb][r], m);
                const int b = cc.b, g = cc.ui / cc.nround;
                const int us = tpre[b] + cc.ui * cc.nt, ue = us + cc.nt;
                if (seg0 == us && t + 1 == ue) {   // the whole unit: write Y
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        float f[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            f[r] = SOFTMAX ? (l_r[nb][r] > 0.f ? 1.f / l_r[nb][r] : 0.f) : 1.f;
                        dec_store_y<D, BF16, DLAY>(p, rr[nb], o[nb], f);
                    }
                } else {
                    // partial (O, m, l): slot 0 of this warp for the range's
                    // first unit, slot 1 for its last
                    auto slot_base = [&](int v) { return (size_t)(v * GRP_WARPS + w) * 2; };
                    const size_t slot = slot_base(vg) + (seg0 == t_begin ? 0 : 1);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        if (!dbg_ok(slot < (size_t)p.dec_slots && p.dec_rows == DR, p.status)) break;
                        dec_store_part<D, DLAY>(part + (slot * DR + 8 * nb) * D, o[nb]);
                        if (lane < 4)
#pragma unroll
                            for (int r = 0; r < 2; ++r)
                                pml[slot * DR + 8 * nb + 2 * lane + r] = make_float2(m_r[nb][r], l_r[nb][r]);
                    }
                    __threadfence();
                    __syncwarp();
                    const int v_lo = group_of(us), v_hi = group_of(ue - 1);
                    const int pidx = ppre[b] + g * cc.nrc + chunk;
                    int tk = 0;
                    if (lane == 0 && dbg_ok(pidx >= 0 && pidx <= p.max_pairs, p.status))
                        tk = atomicAdd(&tickets[pidx], 1);
                    tk = __shfl_sync(0xffffffffu, tk, 0);
                    if (tk == v_hi - v_lo) {   // the last of the chunk's warps: merge
                        __threadfence();
                        constexpr int LPR = 32 / DR, DL = D / LPR, MC = DL < 32 ? DL : 32;
                        const int row = lane / LPR, c0 = (lane % LPR) * DL;
                        // the first group's share is its slot 1 unless the unit
                        // starts its range; every later group's share is its slot 0
                        auto slot_of = [&](int v) -> size_t {
                            return slot_base(v) + ((v == v_lo && range_start(v) != us) ? 1 : 0);
                        };
                        float M = -INFINITY;
                        if (SOFTMAX)
                            for (int v = v_lo; v <= v_hi; ++v)
                                M = fmaxf(M, __ldcg(&pml[slot_of(v) * DR + row].x));
                        const DecRow R = dec_row(p, cc.s, b, g, chunk * DR + row, rows, kv_hi);
#pragma unroll 1
                        for (int h = 0; h < DL / MC; ++h) {
                            float acc[MC];
#pragma unroll
                            for (int k = 0; k < MC; ++k) acc[k] = 0.f;
                            float Lsum = 0.f;
                            for (int v = v_lo; v <= v_hi; ++v) {
                                const size_t sl = slot_of(v);
                                float wt = 1.f;
                                if (SOFTMAX) {
                                    const float2 x = __ldcg(&pml[sl * DR + row]);
                                    wt = (x.x == -INFINITY) ? 0.f : ex2(x.x - M);
                                    Lsum += x.y * wt;
                                }
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    part + (sl * DR + row) * D + c0 + h * MC);
#pragma unroll
                                for (int k = 0; k < MC / 4; ++k) {
                                    const float4 x4 = __ldcg(src + k);
                                    acc[4 * k] += x4.x * wt;
                                    acc[4 * k + 1] += x4.y * wt;
                                    acc[4 * k + 2] += x4.z * wt;
                                    acc[4 * k + 3] += x4.w * wt;
                                }
                            }
                            if (R.valid && dbg_ok(R.qoff >= 0 && R.qoff + D <= q_elems(p), p.status)) {
                                const float f = SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f;
                                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) +
                                                                       R.qoff + c0 + h * MC);
#pragma unroll
                                for (int k = 0; k < MC / 8; ++k)
                                    dst[k] = make_uint4(pack2<BF16>(acc[8 * k] * f, acc[8 * k + 1] * f),
                                                        pack2<BF16>(acc[8 * k + 2] * f, acc[8 * k + 3] * f),
                                                        pack2<BF16>(acc[8 * k + 4] * f, acc[8 * k + 5] * f),
                                                        pack2<BF16>(acc[8 * k + 6] * f, acc[8 * k + 7] * f));
                            }
                        }
                        if (lane == 0) tickets[pidx] = 0;   // ready for the next call
                    }
                }
            }
            advance(cc);
            if (unit_end && t + 1 < t_end) {
                start_unit();
                seg0 = t + 1;
            }
        }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    if (w == 0)
        while (consumed < issued) {
            mbar_wait_drain(&land[consumed % NS], (consumed / NS) & 1);
            ++consumed;
        }
    __syncwarp();
    if (lane == 0 && (!ok || *abort)) set_status(p.status, 5);
}

template <int D, bool BF16, bool SOFTMAX, bool PAGED>
static cudaError_t grp_launch(const AttnParams &p, const TensorMaps &m, cudaStream_t s) {
    using L = GrpLayout<D>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [] {
        return cudaFuncSetAttribute(decode_group_kernel<D, BF16, SOFTMAX, PAGED>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    });
    if (e != cudaSuccess) return e;
    decode_prep_kernel<<<dec_prep_blocks(p), 256, 0, s>>>(p, p.max_pairs + 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_group_kernel<D, BF16, SOFTMAX, PAGED>, p.grid, L::THREADS,
                            L::ALLOC, s, p, m);
}

// Grouped decode over a 16-bit KV cache (p.dec_rows must be DEC_ROWS_WIDE:
// the tickets and partial slots were sized for 16-row chunks, and two slots
// per warp of a grid of p.grid CTAs of 8 warps).
cudaError_t launch_decode_group(const AttnParams &p, const TensorMaps &m, int mode,
                                cudaStream_t s, int bf16) {
    if (p.dec_rows != DEC_ROWS_WIDE || p.dec_slots < 2 * GRP_WARPS * GRP_GROUPS * p.grid)
        return cudaErrorInvalidValue;
    const bool sm = mode == MODE_SOFTMAX;
#define RGA_GRP(D_, B_)                                                                     \
    return p.paged ? (sm ? grp_launch<D_, B_, true, true>(p, m, s)                          \
                         : grp_launch<D_, B_, false, true>(p, m, s))                        \
                   : (sm ? grp_launch<D_, B_, true, false>(p, m, s)                         \
                         : grp_launch<D_, B_, false, false>(p, m, s))
    if (p.D == 64) {
        if (bf16) { RGA_GRP(64, true); }
        RGA_GRP(64, false);
    }
    if (bf16) { RGA_GRP(128, true); }
    RGA_GRP(128, false);
#undef RGA_GRP
}

}  // namespace rga
