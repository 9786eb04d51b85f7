// Multi-token query paged attention on the 5th-generation tensor core
// (tcgen05) for sm_103a: the same operation, work split, partial states and
// merge post-pass as pa_multi_kernel (chunked prefill and speculative
// verification: thewebvale "vLLM & High-Throughput Serving", section 4;
// letsbuildsolutions "How LLM Inference Engines Work", speculative decoding),
// for launches whose (sequence, KV head) pairs carry 17 to 128 query rows.
//
// Tile.  The rows r = i * g + hh of a pair (token i of the chunk, head hh of
// the group) are the M = 128 rows of every MMA; rows past q_len * g are
// computed and discarded (rows are independent in both products).  Keys come
// in stages of 64 (64 / B blocks of one pair).
//
//   S  = Q K^T   M 128, N 64, K = head_dim   (Q, K: K-major swizzled tiles)
//   O += P V     M 128, N = head_dim, K 64   (P: from tensor memory; V:
//                                             MN-major tiles, one per block)
//
// with S (two 64-column fp32 buffers), P (two buffers of 16-bit weights, the
// A operand of the PV product) and O (fp32) all in tensor memory.  P enters
// as a hi + lo pair of 16-bit values (two MMAs), keeping ~16 bits of each
// weight as the mma.sync kernels do.
//
// Warp roles (352 threads, one CTA per SM):
//   warps 0-7  softmax, two streams on alternating stages: warp w takes rows
//              32 (w % 4) .. + 31 (its TMEM lane quarter; thread = query row)
//              of the stages of parity w / 4.  Masks per row (causal limit),
//              runs the online softmax and writes P to tensor memory; zeroes
//              the V rows of a stage past the context; at a segment end loads
//              O and writes the output rows or the partial state.
//   warp 8     copies: per segment the Q tile (one 3-D TMA per 64-column
//              half: box = g heads x max_q tokens, landing as rows i * g + hh);
//              per stage one TMA box per block and operand, issued by
//              different lanes (the TMA unit's cost is per box, so fewer,
//              larger boxes keep more bytes in flight).
//   warp 9     scores: allocates TMEM; one thread issues S of each stage as
//              soon as its copy has landed and its TMEM buffer is free.
//   warp 10    PV: one thread issues the PV product of each stage once its P
//              is written; the commit frees the stage's ring slot.
//
// Lazy rescaling.  A row keeps the reference maximum m_ref used for its
// weights; only when a stage raises the row maximum above m_ref + 8 (log2
// units) is O rescaled in TMEM (after the previous PV completed) and m_ref
// moved.  Weights stay <= 2^8, exact enough in 16 bits with the hi / lo
// split, and O / l is unchanged by the choice of reference.
//
// Hand-offs are mbarriers: full / empty per ring stage, S full / free and
// P full / PV done per TMEM / P buffer, Q full / empty.  Every wait is bounded
// (PA_DEVERR_TIMEOUT, then the CTA drains and releases TMEM); bad block ids
// set PA_DEVERR_BLOCK_ID and poison the segment's rows with NaN.
#pragma once

#include "multi_kernel.cuh"
#include "tc.cuh"

namespace pa {

template <int D_, int BS_, bool BF16_>
struct TcTraits {
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr bool BF16 = BF16_;
    static constexpr int ROWS = 128;                         // M of every MMA
    static constexpr int KEYS = 64;                          // keys per stage (N of the score MMA)
    static constexpr int SB = KEYS / BS;                     // blocks per stage
    static constexpr int HALVES = D / 64;                    // 128-byte column halves of a row
    static constexpr int KV_BYTES = KEYS * D * 2;            // a stage's K, or its V
    // Each block of a stage arrives as one TMA box per operand.
    //  * K: [8-row group][column half][8 rows][128 B] (a 4-D box), so the
    //    8-row groups of one half follow each other HALVES x 1024 bytes apart
    //    across the stage's blocks and the score MMA spans all 64 keys with
    //    one descriptor (that fixed group stride);
    //  * V: [column half][BS rows][128 B] (a 3-D box), an MN-major tile per
    //    block for the PV product.
    static constexpr int GROUP_STRIDE = HALVES * 1024;       // between 8-key groups of K
    static constexpr int HALF_STRIDE = BS * 128;             // between the column halves of a V block tile
    static constexpr int BLK_BYTES = HALVES * HALF_STRIDE;   // one block's K or V tile
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;         // K, then V
    // Shared memory: barriers, stage records, exchange cells and a few words
    // first (sized for R_CAP stages); then the Q tile, as many rows as the
    // launch's chunks fill (q_rows(): the rows past them are read by the score
    // MMA and discarded, whatever they hold); then the ring, as many stages as
    // fit (ring_stages()), so shorter chunks get a deeper ring.
    static constexpr int SMEM_CAP = 227 * 1024;
    static constexpr int SMEM_BYTES = SMEM_CAP;              // all of it, 1024 of it alignment slack
    static constexpr int R_CAP = 12;
    static constexpr int REC_BYTES = 48;
    static constexpr int NBAR_FIXED = 12;    // s_full[2] s_free[2] p_full[2] pv_done[2] q_full q_empty fin o_free
    // tagged cells per row: softmax references along a segment's stages [4],
    // and the partial row sums handed to a segment's last stage [4] (value, reference)
    static constexpr int XCH_BYTES = (4 + 2 * 4) * ROWS * 8;
    static constexpr int BAR_OFF = 0;
    static constexpr int REC_OFF = (BAR_OFF + 8 * (2 * R_CAP + NBAR_FIXED) + 15) / 16 * 16;
    static constexpr int XCH_OFF = REC_OFF + R_CAP * REC_BYTES;
    static constexpr int MISC_OFF = XCH_OFF + XCH_BYTES;      // TMEM base, abort flag, stage count
    static constexpr int Q_OFF = (MISC_OFF + 16 + 1023) / 1024 * 1024;
    // rows of the Q tile: the launch's q_box tokens x g heads, whole 8-row swizzle atoms
    __host__ __device__ static constexpr int q_rows(int q_box, int g) {
        return q_box * g >= ROWS ? ROWS : (q_box * g + 7) / 8 * 8;
    }
    __host__ __device__ static constexpr int ring_stages(int qrows) {
        return (SMEM_CAP - 1024 - Q_OFF - HALVES * qrows * 128) / STAGE_BYTES > R_CAP
                   ? R_CAP
                   : (SMEM_CAP - 1024 - Q_OFF - HALVES * qrows * 128) / STAGE_BYTES;
    }
    static constexpr int SOFT_WARPS = 8;
    static constexpr int THREADS = 32 * (SOFT_WARPS + 3);
    static constexpr int COPY_WARP = SOFT_WARPS, MMA_WARP = SOFT_WARPS + 1, PV_WARP = SOFT_WARPS + 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 128;                        // S buffers at columns 0 and 64
    static constexpr int P_COL = 256;                        // P buffer b at P_COL + 64 b: hi, then lo
    static constexpr int PSTRIDE = D + 4;
    static constexpr float TAU = 8.f;                        // lazy-rescale threshold (log2 units)
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(ring_stages(ROWS) >= 3, "three ring stages at least (the MMA issue order relies on it)");
    static_assert(O_COL + D <= P_COL && P_COL + 128 <= TMEM_COLS, "tensor memory");
};

// One ring stage as the copy warp describes it to the consumers.
struct alignas(16) TcStage {
    int s, kvh, t0, nkeys;       // sequence, KV head, first key, keys copied (blocks x B)
    int n, ctx, q0, flags;       // chunk length, context, first query row of the sequence
    int poison, seg, pad1, pad2;  // bad block id seen; segment number within the CTA
};
static_assert(sizeof(TcStage) == 48, "stage record");

enum : int { TC_FIRST = 1, TC_LAST = 2, TC_COMPLETE = 4, TC_SLOT1 = 8, TC_END = 16, TC_PENULT = 32 };

// A value handed to the other warp of a row quarter: one 64-bit shared word
// holding the value and a tag naming the stage it belongs to, so the reader
// waits (bounded) for that stage's value and never for a barrier.
__device__ __forceinline__ void xch_put(volatile unsigned long long* cell, float v, uint32_t tag) {
    *cell = ((unsigned long long)tag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ bool xch_get(const volatile unsigned long long* cell, uint32_t tag, uint64_t limit_ns,
                                        float& v) {
    unsigned long long x = *cell;
    if ((uint32_t)(x >> 32) != tag) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 1;; ++i) {
            x = *cell;
            if ((uint32_t)(x >> 32) == tag) break;
            if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
        }
    }
    v = __uint_as_float((uint32_t)x);
    return true;
}

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, 1)
pa_multi_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const MultiParams mp) {
    constexpr int D = Tr::D, BS = Tr::BS, SB = Tr::SB, HALVES = Tr::HALVES, KEYS = Tr::KEYS;
    constexpr int SW = Tr::SOFT_WARPS;
    constexpr uint32_t IDESC_S = idesc_f16<Tr::BF16>(128, KEYS, false, false);
    constexpr uint32_t IDESC_O = idesc_f16<Tr::BF16>(128, D, false, true);
    const DecodeParams& p = mp.d;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;
    const uint32_t sbase = smem_u32(smem);
    const int qrows = Tr::q_rows(mp.q_box, G);
    const uint32_t q_half = (uint32_t)qrows * 128;            // between the Q tile's column halves
    const int R = Tr::ring_stages(qrows);                     // ring stages
    const uint32_t q_tile = sbase + Tr::Q_OFF;
    const uint32_t ring_off = Tr::Q_OFF + HALVES * q_half;
    const uint32_t ring = sbase + ring_off;
    const uint32_t bars = sbase + Tr::BAR_OFF;
    auto full = [&](int st) -> uint32_t { return bars + 8 * st; };
    auto empty = [&](int st) -> uint32_t { return bars + 8 * (R + st); };
    const uint32_t s_full = bars + 16 * R, s_free = s_full + 16, p_full = s_free + 16, pv_done = p_full + 16;
    const uint32_t q_full = pv_done + 16, q_empty = q_full + 8, fin = q_empty + 8, o_free = fin + 8;
    TcStage* recs = reinterpret_cast<TcStage*>(smem + Tr::REC_OFF);
    volatile unsigned long long* xch = reinterpret_cast<volatile unsigned long long*>(smem + Tr::XCH_OFF);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Tr::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Tr::MISC_OFF + 4);
    volatile int* n_stages = reinterpret_cast<volatile int*>(smem + Tr::MISC_OFF + 8);   // set at the end record

    if (threadIdx.x == 0) {
        for (int st = 0; st < R; ++st) {
            mbar_init(full(st), 1);
            mbar_init(empty(st), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + 8 * b, 1);
            mbar_init(s_free + 8 * b, SW / 2);      // the four warps of the stage's stream
            mbar_init(p_full + 8 * b, SW / 2);
            mbar_init(pv_done + 8 * b, 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(fin, 2);                      // the score thread and the PV thread
        mbar_init(o_free, SW / 2);              // a segment's output read: the four warps of its last stage
        *abort_flag = 0;
        *n_stages = 0x7fffffff;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < Tr::XCH_BYTES / 8; i += Tr::THREADS) xch[i] = 0ull;   // tag 0: nothing yet
    if (warp == Tr::MMA_WARP) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), Tr::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == Tr::COPY_WARP && lane == 0) {
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched with programmatic stream serialization after the pre-pass:
    // the set-up above overlaps it; nothing the stream wrote is read before
    // it completes.  The merge post-pass may then be placed as CTAs retire.
    griddep_wait();
    griddep_launch_dependents();

    SeqTab tab;
    tab.cum = p.cum;
    tab.ctx = p.context_lens;
    tab.first = nullptr;
    const int32_t* qst = mp.q_start;
    // a sequence's chunk length, or -1 when it is malformed
    auto chunk_len = [&](int s) -> int {
        const int a = __ldg(qst + s), b = __ldg(qst + s + 1), ctx = __ldg(p.context_lens + s);
        const int n = b - a;
        const bool ok = a >= 0 && b <= mp.total_q && n >= 0 && n <= mp.max_q && n <= (ctx > 0 ? ctx : 0);
        return ok ? n : -1;
    };

    // ---- malformed chunks and bad context lengths: error bit, NaN rows ----
    for (int s = blockIdx.x; s < p.N; s += gridDim.x) {
        const int n = chunk_len(s);
        const int ctx = __ldg(p.context_lens + s);
        const bool bad_ctx = ctx < 0 || ctx > p.MB * BS;
        if (n >= 0 && !bad_ctx) continue;
        if (threadIdx.x == 0) set_err(p.err, PA_DEVERR_CONTEXT);
        const int a = max(0, __ldg(qst + s));
        const int b = min(mp.total_q, __ldg(qst + s + 1));
        for (long long i = (long long)a * p.Hq * D + threadIdx.x; i < (long long)b * p.Hq * D; i += Tr::THREADS)
            p.out[i] = qnan16<Tr::BF16>();
    }

    const Sched sc = make_sched(__ldg(p.cum + p.N) * p.Hkv, gridDim.x, 0);
    const bool has_work = (int)blockIdx.x < sc.NS;
    const long long lo = has_work ? sc.lo(blockIdx.x) : 0, hi = has_work ? sc.lo(blockIdx.x + 1) : 0;

    if (warp == Tr::COPY_WARP) {
        const uint64_t kv_pol = l2_evict_first();
        // ================================================================ copies
        int j = 0, st = 0, nseg = 0;            // stage, its ring slot and phase
        uint32_t ph = 0;
        bool ok = true;
        auto claim = [&]() -> bool {            // lane 0: slot st free for stage j (its last use done)
            return j < R || mbar_wait_bounded(empty(st), ph ^ 1u, p.timeout_ns);
        };
        if (has_work) {
            SegIter it = locate(p, tab, lo, lane);
            while (ok && it.gi < hi) {
                const int len = seg_len(it, hi);
                const int n = chunk_len(it.s);
                if (n > 0) {
                    const int ctx = __ldg(p.context_lens + it.s);
                    const int q0 = __ldg(qst + it.s);
                    const long long P0 = it.gi - it.b0;
                    const bool complete = sc.of(P0) == sc.of(P0 + it.nb - 1);
                    const int seg_flags = (complete ? TC_COMPLETE : 0) | (it.gi == lo ? 0 : TC_SLOT1);
                    if (lane == 0) {
                        if (nseg > 0 && !mbar_wait_bounded(q_empty, (uint32_t)((nseg - 1) & 1), p.timeout_ns)) {
                            ok = false;
                        } else {
                            mbar_arrive_expect_tx(q_full, (uint32_t)(HALVES * 128 * G * mp.q_box));
#pragma unroll
                            for (int h = 0; h < HALVES; ++h)
                                tma_load_3d(q_tile + h * q_half, &tmap_q, h * 64, it.kvh * G, q0, q_full);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    ++nseg;
                    const int32_t* trow = p.block_tables + (size_t)it.s * p.MB + it.b0;
                    auto batch = [&](int from) -> int { return lane < len - from ? __ldg(trow + from + lane) : 0; };
                    int ids = batch(0), ids_next = batch(32);
                    const int nst = (len + SB - 1) / SB;
                    for (int k = 0; ok && k < nst; ++k) {
                        const int bb = k * SB;
                        if (bb > 0 && (bb & 31) == 0) {
                            ids = ids_next;
                            ids_next = batch(bb + 32);
                        }
                        const int nbs = min(SB, len - bb);
                        int idv[SB];
#pragma unroll
                        for (int i = 0; i < SB; ++i) idv[i] = __shfl_sync(0xffffffffu, ids, (bb + i) & 31);
                        if (lane == 0) {
                            if (!claim()) {
                                ok = false;
                            } else {
                                int poison = 0;
#pragma unroll
                                for (int i = 0; i < SB; ++i)
                                    if (i < nbs && (unsigned)idv[i] >= (unsigned)p.NB) {
                                        poison = 1;
                                        idv[i] = 0;
                                    }
                                if (poison) set_err(p.err, PA_DEVERR_BLOCK_ID);
                                TcStage& rc = recs[st];
                                rc.s = it.s;
                                rc.kvh = it.kvh;
                                rc.t0 = (it.b0 + bb) * BS;
                                rc.nkeys = nbs * BS;
                                rc.n = n;
                                rc.ctx = ctx;
                                rc.q0 = q0;
                                rc.flags = seg_flags | (k == 0 ? TC_FIRST : 0) | (k == nst - 1 ? TC_LAST : 0) |
                                           (k == nst - 2 ? TC_PENULT : 0);
                                rc.poison = poison;
                                rc.seg = nseg;
                                mbar_arrive_expect_tx(full(st), (uint32_t)(nbs * BS * 128 * HALVES * 2));
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        __syncwarp();   // lane 0's claim of the slot orders the other lanes' copies
                        // the stage's copies, one box per lane (the TMA unit takes boxes
                        // one at a time, so each block's K and V go as one box each):
                        // lanes 0 .. SB - 1 the K boxes, the next SB lanes the V boxes
                        {
                            const bool kl = lane < SB;
                            const int ci = kl ? lane : lane - SB;
                            int cid = __shfl_sync(0xffffffffu, ids, (bb + (ci & (SB - 1))) & 31);
                            if ((unsigned)cid >= (unsigned)p.NB) cid = 0;   // flagged and poisoned above
                            const int y = (cid * p.Hkv + it.kvh) * BS;
                            const uint32_t dst = ring + st * Tr::STAGE_BYTES + (kl ? 0 : Tr::KV_BYTES) + ci * Tr::BLK_BYTES;
                            if (ok && lane < 2 * SB && ci < nbs) {
                                // each block is read once: L2 evict-first
                                if (kl)
                                    tma_load_4d_hint(dst, &tmap_k, 0, 0, 0, y / 8, full(st), kv_pol);
                                else
                                    tma_load_3d_hint(dst, &tmap_v, 0, y, 0, full(st), kv_pol);
                            }
                        }
                        ++j;
                        if (++st == R) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                }
                seg_advance(it, len, p, tab);
            }
        }
        if (lane == 0) {
            // the end record, twice: each softmax stream takes every other stage
            for (int e = 0; e < 2 && ok; ++e) {
                if (claim()) {
                    recs[st].flags = TC_END;
                    mbar_arrive(full(st));
                    ++j;
                    if (++st == R) {
                        st = 0;
                        ph ^= 1u;
                    }
                } else {
                    ok = false;
                }
            }
            if (!ok) {
                set_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
                // copies still in flight land before the CTA's shared memory is released
                for (int k = j - R > 0 ? j - R : 0; k < j; ++k)
                    mbar_wait_bounded(full(k % R), (uint32_t)((k / R) & 1), p.timeout_ns);
                if (nseg > 0) mbar_wait_bounded(q_full, (uint32_t)((nseg - 1) & 1), p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == Tr::MMA_WARP) {
        // ================================================================ scores
        // One thread issues S_j as soon as its inputs are ready: the copy of
        // stage j, the scores of stage j - 2 read out of its TMEM buffer
        // (s_free) and, at a segment start, the Q tile.  The PV products are
        // issued by another thread (PV_WARP), so neither kind of MMA waits
        // behind the other's inputs.  At the end record it publishes the
        // number of stages.  No progress for the wait limit: abort.
        if (lane == 0) {
            int js = 0, nseg = 0;                        // next S, Q tiles consumed
            int s_st = 0;                                // ring slot and phase of stage js
            uint32_t s_ph = 0;
            bool ok = true;
            uint64_t t_last = global_timer_ns();
            for (uint32_t spin = 0;; ++spin) {
                if (mbar_test_wait(full(s_st), s_ph)) {
                    const int flags = recs[s_st].flags;
                    if (flags & TC_END) {
                        *n_stages = js;
                        break;
                    }
                    if ((!(flags & TC_FIRST) || mbar_test_wait(q_full, (uint32_t)(nseg & 1))) &&
                        (js < 2 || mbar_test_wait(s_free + 8 * (js & 1), (uint32_t)(((js - 2) >> 1) & 1)))) {
                        const int b = js & 1;
                        if (flags & TC_FIRST) ++nseg;
                        tc_fence_after();
                        const uint64_t qd = sdesc_sw128(q_tile, 16, 1024);
                        const uint64_t kd = sdesc_sw128(ring + s_st * Tr::STAGE_BYTES, 16, Tr::GROUP_STRIDE);
#pragma unroll
                        for (int k = 0; k < D / 16; ++k) {      // +32 bytes per K step; per 4: Q's next half tile,
                                                                // K's next 1024-byte atom (address >> 4)
                            mma_f16(tmem + 64 * b, qd + (uint64_t)((k / 4) * (q_half >> 4) + (k % 4) * 2),
                                    kd + (uint64_t)((k / 4) * (1024 >> 4) + (k % 4) * 2), IDESC_S,
                                    k > 0 ? 1u : 0u);
                        }
                        mma_commit(s_full + 8 * b);
                        if (flags & TC_LAST) mma_commit(q_empty);
                        ++js;
                        if (++s_st == R) {
                            s_st = 0;
                            s_ph ^= 1u;
                        }
                        t_last = global_timer_ns();
                        continue;
                    }
                }
                if ((spin & 63u) == 0 && (*abort_flag || global_timer_ns() - t_last > p.timeout_ns)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                set_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued (by both threads) completes before tensor memory is released
            mma_commit(fin);
            mbar_wait_bounded(fin, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == Tr::PV_WARP) {
        // ================================================================ PV
        // One thread issues PV_j in stage order once P_j is written and, at a
        // segment start, the previous segment's output has been read; the
        // commit frees the stage's ring slot.  It stops at the number of
        // stages the score thread publishes.
        if (lane == 0) {
            int jp = 0, pv_seg = 0;
            bool ok = true;
            while (true) {
                const int b = jp & 1;
                bool ready = false;
                const uint64_t t0 = global_timer_ns();
                for (uint32_t spin = 0;; ++spin) {
                    if (jp >= *n_stages) break;
                    if (mbar_test_wait(p_full + 8 * b, (uint32_t)((jp >> 1) & 1))) {
                        ready = true;
                        break;
                    }
                    if ((spin & 63u) == 0 && (*abort_flag || global_timer_ns() - t0 > p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                }
                if (!ready) break;
                const int st = jp % R;
                const bool first = (recs[st].flags & TC_FIRST) != 0;
                // a segment's first PV overwrites O: the previous segment's output must have been read
                if (first && pv_seg > 0 && !mbar_wait_bounded(o_free, (uint32_t)((pv_seg - 1) & 1), p.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (first) ++pv_seg;
                tc_fence_after();
                const uint32_t pt = tmem + Tr::P_COL + 64 * b;
                const uint32_t vbase = ring + st * Tr::STAGE_BYTES + Tr::KV_BYTES;
#pragma unroll
                for (int k = 0; k < KEYS / 16; ++k) {
                    // keys 16 k .. 16 k + 15: rows (16 k) % BS .. of block tile (16 k) / BS
                    const uint64_t bv = sdesc_sw128(vbase + ((16 * k) / BS) * Tr::BLK_BYTES + ((16 * k) % BS) * 128,
                                                    Tr::HALF_STRIDE, 1024);
                    mma_f16_ts(tmem + Tr::O_COL, pt + 8 * k, bv, IDESC_O, (first && k == 0) ? 0u : 1u);
                    mma_f16_ts(tmem + Tr::O_COL, pt + 32 + 8 * k, bv, IDESC_O, 1u);
                }
                mma_commit(pv_done + 8 * b);
                mma_commit(empty(st));
                ++jp;
            }
            if (!ok) {
                set_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            mma_commit(fin);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax
        // Warp w takes rows 32 (w % 4) .. + 31 (its TMEM lane quarter; thread =
        // query row) of every other stage: stream w / 4 takes the stages of its
        // parity, so the two warps of a lane quarter work on consecutive stages
        // at once.  Per row, the softmax reference is handed along a segment's
        // stages (a tagged cell, written once the stage's maximum is known); each
        // stream keeps its own partial row sum, and the segment's last stage adds
        // the other stream's.  O is one accumulator: a stage that moves the
        // reference rescales it after the previous stage's PV has completed.
        const int quarter = warp & 3, stream = warp >> 2;
        const int r = quarter * 32 + lane;                      // query row = TMEM lane
        const int stid = quarter * 32 + lane;                   // thread index within the stream
        // bounded wait whose outcome is the same on every lane of the warp
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, p.timeout_ns));
        };
        auto get_all = [&](const volatile unsigned long long* cell, uint32_t tag, float& v) -> bool {
            return __all_sync(0xffffffffu, xch_get(cell, tag, p.timeout_ns, v));
        };
        volatile unsigned long long* ref_cell = xch;                      // [4][ROWS] by tag % 4
        volatile unsigned long long* sum_cell = xch + 4 * Tr::ROWS;       // [4][ROWS] partial sums by segment % 4
        volatile unsigned long long* sref_cell = xch + 8 * Tr::ROWS;      // [4][ROWS] their references
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t o_addr = lane_addr + Tr::O_COL;
        const float qnan = __int_as_float(0x7fc00000);
        int j = stream, st = stream;                            // this stream's stage, its ring slot and phase
        uint32_t ph = 0;
        float m_mine = -INFINITY, l = 0.f;                      // reference of this stream's sum, the sum
        int pois = 0, lim = -1, cur_seg = -1, seg_kvh = 0, seg_q0 = 0;
        bool wact = false, ok = true;
        while (true) {
            if (*abort_flag) break;
            if (!wait_all(full(st), ph)) {
                ok = false;
                break;
            }
            const int flags = recs[st].flags;
            if (flags & TC_END) break;
            const int t0 = recs[st].t0, nkeys = recs[st].nkeys, ctx = recs[st].ctx, seg = recs[st].seg;
            if (seg != cur_seg) {
                const int n = recs[st].n;
                cur_seg = seg;
                seg_kvh = recs[st].kvh;
                seg_q0 = recs[st].q0;
                m_mine = -INFINITY;
                l = 0.f;
                pois = 0;
                lim = r < n * G ? ctx - n + r / G : -1;
                wact = __any_sync(0xffffffffu, lim >= 0);
            }
            pois |= recs[st].poison;
            const int b = j & 1;
            // P buffer b is free once this stream's previous PV is done.  Every warp
            // of the stream waits for it before arriving for this stage, active or
            // not: a warp that skipped ahead could otherwise count toward the
            // previous stage's P-ready phase before that stage's P was written.
            bool p_free = j < 2;
            auto p_buffer_free = [&]() -> bool {
                if (!p_free) p_free = wait_all(pv_done + 8 * b, (uint32_t)(((j - 2) >> 1) & 1));
                return p_free;
            };
            if (!wait_all(s_full + 8 * b, (uint32_t)((j >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[KEYS];
            if (wact) {
                uint32_t u0[32], u1[32];
                tmem_ld32(lane_addr + 64 * b, u0);
                tmem_ld32(lane_addr + 64 * b + 32, u1);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    x[k] = __uint_as_float(u0[k]);
                    x[32 + k] = __uint_as_float(u1[k]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free + 8 * b);
            if (wact) {
                const int kv = min(nkeys, max(0, lim - t0 + 1));   // keys this row sees here
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (__all_sync(0xffffffffu, kv >= KEYS)) {
#pragma unroll
                    for (int k = 0; k < KEYS; ++k) {
                        x[k] *= p.scale_log2;
                        m4[k & 3] = fmaxf(m4[k & 3], x[k]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < KEYS; ++k) {
                        x[k] = k < kv ? x[k] * p.scale_log2 : -INFINITY;
                        m4[k & 3] = fmaxf(m4[k & 3], x[k]);
                    }
                }
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                // the reference after the previous stage of the segment (other stream)
                float m_prev = -INFINITY;
                if (!(flags & TC_FIRST) && !get_all(ref_cell + (j & 3) * Tr::ROWS + r, (uint32_t)j, m_prev)) {
                    ok = false;
                    break;
                }
                if (m_prev != m_mine) {                      // references only grow along a segment
                    l *= m_mine == -INFINITY ? 0.f : ex2(m_mine - m_prev);
                    m_mine = m_prev;
                }
                const float m_new = fmaxf(m_prev, mx);
                const bool need = m_new > m_prev + Tr::TAU;
                if (need) m_mine = m_new;
                if (!(flags & TC_LAST)) xch_put(ref_cell + ((j + 1) & 3) * Tr::ROWS + r, m_mine, (uint32_t)(j + 1));
                const float alpha = need ? ex2(m_prev - m_new) : 1.f;      // m_prev = -inf: 0
                if (need) l *= alpha;
                if (!(flags & TC_FIRST) && __any_sync(0xffffffffu, need)) {
                    // O holds the earlier stages once the previous stage's PV is done
                    if (!wait_all(pv_done + 8 * (b ^ 1), (uint32_t)(((j - 1) >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t u[32];
                        tmem_ld32(o_addr + 32 * c, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
                        tmem_st32(o_addr + 32 * c, u);
                    }
                    tmem_st_wait();
                }
                const float mref = m_mine == -INFINITY ? 0.f : m_mine;      // no visible key yet: weights 0
                if (!p_buffer_free()) {
                    ok = false;
                    break;
                }
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 2; ++c) {            // 32 keys at a time: hi, lo columns 16 c ..
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = ex2(x[32 * c + 2 * e] - mref), p1 = ex2(x[32 * c + 2 * e + 1] - mref);
                        s4[e & 3] += p0 + p1;
                        if constexpr (Tr::BF16) {
                            // hi: the weights cut to bf16 (their top 16 bits); lo: the exact
                            // remainders, cut the same way (relative error < 2^-14 in all)
                            const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
                            hw[e] = __byte_perm(u0, u1, 0x7632);
                            const float r0 = p0 - __uint_as_float(u0 & 0xffff0000u);
                            const float r1 = p1 - __uint_as_float(u1 & 0xffff0000u);
                            lw[e] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
                        } else {
                            const uint32_t hv = pack2<false>(p0, p1);
                            hw[e] = hv;
                            lw[e] = pack2<false>(p0 - lo_of<false>(hv), p1 - hi_of<false>(hv));
                        }
                    }
                    tmem_st16(lane_addr + Tr::P_COL + 64 * b + 16 * c, hw);
                    tmem_st16(lane_addr + Tr::P_COL + 64 * b + 32 + 16 * c, lw);
                }
                l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
            // V rows past the context or past the blocks copied are zero for the PV product
            const int vvalid = max(0, min(nkeys, ctx - t0));
            if (vvalid < KEYS) {
                uint8_t* vt = smem + ring_off + st * Tr::STAGE_BYTES + Tr::KV_BYTES;
                const int nz = (KEYS - vvalid) * HALVES * 8;
                for (int i = stid; i < nz; i += 128) {
                    const int key = vvalid + i / (HALVES * 8), part = i % (HALVES * 8);
                    *reinterpret_cast<uint4*>(vt + (key / BS) * Tr::BLK_BYTES + (part / 8) * Tr::HALF_STRIDE +
                                              (key % BS) * 128 + (part % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            if (!p_buffer_free()) {
                ok = false;
                break;
            }
            if (wact) tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + 8 * b);
            if ((flags & TC_PENULT) && wact) {
                // this stream's share of the row sums, for the segment's last stage
                xch_put(sum_cell + (seg & 3) * Tr::ROWS + r, l, (uint32_t)(seg + 1));
                xch_put(sref_cell + (seg & 3) * Tr::ROWS + r, m_mine, (uint32_t)(seg + 1));
            }
            if (flags & TC_LAST) {
                if (!wait_all(pv_done + 8 * b, (uint32_t)((j >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (wact) {
                    float L = l;
                    if (!(flags & TC_FIRST)) {
                        float l2 = 0.f, m2 = -INFINITY;
                        if (!get_all(sum_cell + (seg & 3) * Tr::ROWS + r, (uint32_t)(seg + 1), l2) ||
                            !get_all(sref_cell + (seg & 3) * Tr::ROWS + r, (uint32_t)(seg + 1), m2)) {
                            ok = false;
                            break;
                        }
                        if (m2 != -INFINITY) L += l2 * ex2(m2 - m_mine);
                    }
                    const bool live = lim >= 0;
                    if (flags & TC_COMPLETE) {
                        uint16_t* orow = p.out + ((size_t)(seg_q0 + r / G) * p.Hq + (size_t)seg_kvh * G + r % G) * D;
                        const float inv = 1.f / L;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t u[32];
                            tmem_ld32(o_addr + 32 * c, u);
                            tmem_ld_wait();
                            uint32_t w[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const float o0 = pois ? qnan : __uint_as_float(u[2 * k]) * inv;
                                const float o1 = pois ? qnan : __uint_as_float(u[2 * k + 1]) * inv;
                                w[k] = pack2<Tr::BF16>(o0, o1);
                            }
                            if (live) {
                                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                            }
                        }
                    } else {
                        float* prow = p.partials +
                                      (((size_t)blockIdx.x * 2 + ((flags & TC_SLOT1) ? 1 : 0)) * Tr::ROWS + r) *
                                          Tr::PSTRIDE;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t u[32];
                            tmem_ld32(o_addr + 32 * c, u);
                            tmem_ld_wait();
                            if (live) {
                                float4* dst = reinterpret_cast<float4*>(prow + 32 * c);
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    float4 v;
                                    v.x = pois ? qnan : __uint_as_float(u[4 * k]);
                                    v.y = pois ? qnan : __uint_as_float(u[4 * k + 1]);
                                    v.z = pois ? qnan : __uint_as_float(u[4 * k + 2]);
                                    v.w = pois ? qnan : __uint_as_float(u[4 * k + 3]);
                                    dst[k] = v;
                                }
                            }
                        }
                        if (live) {
                            prow[D] = m_mine;
                            prow[D + 1] = L;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
            }
            j += 2;
            st += 2;
            if (st >= R) {
                st -= R;
                ph ^= 1u;
            }
        }
        if (!ok) {
            if (lane == 0) set_err(p.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == Tr::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, Tr::TMEM_COLS);
    }
}

template <class Tr>
cudaError_t multi_tc_launch(const MultiLaunch& L) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream, attr);
    return cudaLaunchKernelEx(&cfg, pa_multi_tc_kernel<Tr>, *L.tmap_q, *L.tmap_k, *L.tmap_v, L.p);
}

template <class Tr>
MultiKernelInfo multi_tc_info() {
    return MultiKernelInfo{&multi_tc_launch<Tr>,
                           &persistent_ctas<pa_multi_tc_kernel<Tr>, Tr::THREADS, Tr::SMEM_BYTES>, Tr::ROWS};
}

// Index: [bs == 32]; one table per (dtype, head_dim), defined in multi_tc_*.cu.
void multi_tc_table_bf16_d128(MultiKernelInfo (&t)[2]);
void multi_tc_table_bf16_d64(MultiKernelInfo (&t)[2]);
void multi_tc_table_fp16_d128(MultiKernelInfo (&t)[2]);
void multi_tc_table_fp16_d64(MultiKernelInfo (&t)[2]);

}  // namespace pa
