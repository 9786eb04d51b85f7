// Multi-token query paged attention on the 5th-generation tensor core
// (tcgen05) for sm_103a: the same operation, work split, partial states and
// merge post-pass as pa_multi_kernel (chunked prefill and speculative
// verification: thewebvale "vLLM & High-Throughput Serving", section 4;
// letsbuildsolutions "How LLM Inference Engines Work", speculative decoding),
// for launches whose (sequence, KV head) pairs carry up to 128 query rows.
//
// Tile.  The rows r = i * g + hh of a pair (token i of the chunk, head hh of
// the group) are the M = 128 rows of every MMA; rows past q_len * g are
// computed and discarded (rows are independent in both products).  Keys come
// in stages of 64 (64 / B blocks of one pair).
//
//   S  = Q K^T   M 128, N 64, K = head_dim   (Q, K: K-major swizzled tiles)
//   O += P V     M 128, N = head_dim, K 64   (P: K-major; V: MN-major tile)
//
// with S (two 64-column buffers) and O (fp32) in tensor memory.  P enters as
// a hi + lo pair of 16-bit values (two MMAs), keeping ~16 bits of each weight
// as the mma.sync kernels do.
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3  softmax: thread = query row = TMEM lane.  Loads the stage's
//              scores, masks per row (causal limit), runs the online softmax
//              and writes P to shared memory; zeroes the V rows of a stage
//              past the context; at a segment end loads O and writes the
//              output rows or the partial state.
//   warp 4     copies: per segment the Q tile (one 3-D TMA per 64-column
//              half: box = g heads x max_q tokens, landing as rows i * g + hh),
//              per stage the K and V boxes of its blocks (2-D TMA).
//   warp 5     MMA: allocates TMEM; issues S of stage j + 1 before PV of
//              stage j so the softmax of one stage overlaps the tensor core.
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
    static constexpr int Q_HALF = ROWS * 128;
    static constexpr int Q_BYTES = HALVES * Q_HALF;
    static constexpr int HALF_BYTES = KEYS * 128;            // one column half of a stage's K or V
    static constexpr int KV_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;         // K, then V
    static constexpr int P_TILE = ROWS * 128;                // 64 16-bit weights per row
    static constexpr int P_OFF = Q_BYTES;                    // [buffer][hi, lo] tiles
    static constexpr int RING_OFF = P_OFF + 4 * P_TILE;
    static constexpr int SMEM_CAP = 227 * 1024;
    static constexpr int REC_BYTES = 48;
    static constexpr int NBAR_FIXED = 11;                    // s_full[2] s_free[2] p_full[2] pv_done[2] q_full q_empty fin
    static constexpr int R_FIT = (SMEM_CAP - 1024 - RING_OFF - 8 * (16 + NBAR_FIXED) - 8 * REC_BYTES - 16) /
                                 STAGE_BYTES;
    static constexpr int R = R_FIT > 8 ? 8 : R_FIT;
    static constexpr int BAR_OFF = RING_OFF + R * STAGE_BYTES;
    static constexpr int REC_OFF = (BAR_OFF + 8 * (2 * R + NBAR_FIXED) + 15) / 16 * 16;
    static constexpr int MISC_OFF = REC_OFF + R * REC_BYTES;  // TMEM base, abort flag
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;   // + alignment slack
    static constexpr int THREADS = 192;
    static constexpr int TMEM_COLS = 256;                    // S buffers at columns 0 and 64, O at 128
    static constexpr int O_COL = 128;
    static constexpr int PSTRIDE = D + 4;
    static constexpr float TAU = 8.f;                        // lazy-rescale threshold (log2 units)
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(R >= 2, "two ring stages at least");
    static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory");
    static_assert(O_COL + D <= TMEM_COLS, "tensor memory");
};

// One ring stage as the copy warp describes it to the consumers.
struct alignas(16) TcStage {
    int s, kvh, t0, nkeys;       // sequence, KV head, first key, keys copied (blocks x B)
    int n, ctx, q0, flags;       // chunk length, context, first query row of the sequence
    int poison, pad0, pad1, pad2;
};
static_assert(sizeof(TcStage) == 48, "stage record");

enum : int { TC_FIRST = 1, TC_LAST = 2, TC_COMPLETE = 4, TC_SLOT1 = 8, TC_END = 16 };

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, 1)
pa_multi_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const MultiParams mp) {
    constexpr int D = Tr::D, BS = Tr::BS, R = Tr::R, SB = Tr::SB, HALVES = Tr::HALVES, KEYS = Tr::KEYS;
    constexpr uint32_t IDESC_S = idesc_f16<Tr::BF16>(128, KEYS, false, false);
    constexpr uint32_t IDESC_O = idesc_f16<Tr::BF16>(128, D, false, true);
    const DecodeParams& p = mp.d;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_tile = sbase;
    const uint32_t p_tiles = sbase + Tr::P_OFF;
    const uint32_t ring = sbase + Tr::RING_OFF;
    const uint32_t bars = sbase + Tr::BAR_OFF;
    auto full = [&](int st) -> uint32_t { return bars + 8 * st; };
    auto empty = [&](int st) -> uint32_t { return bars + 8 * (R + st); };
    const uint32_t s_full = bars + 16 * R, s_free = s_full + 16, p_full = s_free + 16, pv_done = p_full + 16;
    const uint32_t q_full = pv_done + 16, q_empty = q_full + 8, fin = q_empty + 8;
    TcStage* recs = reinterpret_cast<TcStage*>(smem + Tr::REC_OFF);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Tr::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Tr::MISC_OFF + 4);

    if (threadIdx.x == 0) {
        for (int st = 0; st < R; ++st) {
            mbar_init(full(st), 1);
            mbar_init(empty(st), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + 8 * b, 1);
            mbar_init(s_free + 8 * b, 4);
            mbar_init(p_full + 8 * b, 4);
            mbar_init(pv_done + 8 * b, 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), Tr::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

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

    if (warp == 4) {
        // ================================================================ copies
        long long j = 0;
        int nseg = 0;
        bool ok = true;
        auto claim = [&](int st) -> bool {      // lane 0: slot st free for stage j
            return j < R || mbar_wait_bounded(empty(st), (uint32_t)(((j / R) - 1) & 1), p.timeout_ns);
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
                                tma_load_3d(q_tile + h * Tr::Q_HALF, &tmap_q, h * 64, it.kvh * G, q0, q_full);
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
                        const int st = (int)(j % R);
                        if (lane == 0) {
                            if (!claim(st)) {
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
                                rc.flags = seg_flags | (k == 0 ? TC_FIRST : 0) | (k == nst - 1 ? TC_LAST : 0);
                                rc.poison = poison;
                                const uint32_t dst = ring + st * Tr::STAGE_BYTES;
                                mbar_arrive_expect_tx(full(st), (uint32_t)(nbs * BS * 128 * HALVES * 2));
#pragma unroll
                                for (int i = 0; i < SB; ++i) {
                                    if (i >= nbs) break;
                                    const int y = (idv[i] * p.Hkv + it.kvh) * BS;
#pragma unroll
                                    for (int h = 0; h < HALVES; ++h) {
                                        const uint32_t off = h * Tr::HALF_BYTES + i * BS * 128;
                                        tma_load_2d(dst + off, &tmap_k, h * 64, y, full(st));
                                        tma_load_2d(dst + Tr::KV_BYTES + off, &tmap_v, h * 64, y, full(st));
                                    }
                                }
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        ++j;
                    }
                }
                seg_advance(it, len, p, tab);
            }
        }
        if (lane == 0) {
            if (ok) {
                const int st = (int)(j % R);
                if (claim(st)) {
                    recs[st].flags = TC_END;
                    mbar_arrive(full(st));
                } else {
                    ok = false;
                }
            }
            if (!ok) {
                set_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
                // copies still in flight land before the CTA's shared memory is released
                for (long long k = j - R > 0 ? j - R : 0; k < j; ++k)
                    mbar_wait_bounded(full((int)(k % R)), (uint32_t)((k / R) & 1), p.timeout_ns);
                if (nseg > 0) mbar_wait_bounded(q_full, (uint32_t)((nseg - 1) & 1), p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ================================================================ MMA
        if (lane == 0) {
            long long j = 0, pend = -1;
            int nseg = 0, pend_st = 0, pend_first = 0;
            bool ok = true;
            auto issue_pv = [&]() -> bool {
                const int b = (int)(pend & 1);
                if (!mbar_wait_bounded(p_full + 8 * b, (uint32_t)((pend >> 1) & 1), p.timeout_ns)) return false;
                tc_fence_after();
                const uint32_t pa = p_tiles + b * 2 * Tr::P_TILE;
                const uint32_t vb = ring + pend_st * Tr::STAGE_BYTES + Tr::KV_BYTES;
#pragma unroll
                for (int k = 0; k < KEYS / 16; ++k) {
                    const uint64_t bv = sdesc_sw128(vb + k * 16 * 128, Tr::HALF_BYTES, 1024);
                    mma_f16(tmem + Tr::O_COL, sdesc_sw128(pa + k * 32, 16, 1024), bv, IDESC_O,
                            (pend_first && k == 0) ? 0u : 1u);
                    mma_f16(tmem + Tr::O_COL, sdesc_sw128(pa + Tr::P_TILE + k * 32, 16, 1024), bv, IDESC_O, 1u);
                }
                mma_commit(pv_done + 8 * b);
                mma_commit(empty(pend_st));
                pend = -1;
                return true;
            };
            while (true) {
                if (*abort_flag) break;
                const int st = (int)(j % R);
                if (!mbar_wait_bounded(full(st), (uint32_t)((j / R) & 1), p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int flags = recs[st].flags;
                if (flags & TC_END) break;
                if (flags & TC_FIRST) {
                    if (pend >= 0 && !issue_pv()) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded(q_full, (uint32_t)(nseg & 1), p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    ++nseg;
                }
                const int b = (int)(j & 1);
                if (j >= 2 && !mbar_wait_bounded(s_free + 8 * b, (uint32_t)(((j - 2) >> 1) & 1), p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = ring + st * Tr::STAGE_BYTES;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = sdesc_sw128(q_tile + (k / 4) * Tr::Q_HALF + (k % 4) * 32, 16, 1024);
                    const uint64_t bk = sdesc_sw128(kb + (k / 4) * Tr::HALF_BYTES + (k % 4) * 32, 16, 1024);
                    mma_f16(tmem + 64 * b, a, bk, IDESC_S, k > 0 ? 1u : 0u);
                }
                mma_commit(s_full + 8 * b);
                if (flags & TC_LAST) mma_commit(q_empty);
                if (pend >= 0 && !issue_pv()) {
                    ok = false;
                    break;
                }
                pend = j;
                pend_st = st;
                pend_first = (flags & TC_FIRST) != 0;
                ++j;
            }
            if (ok && pend >= 0 && !issue_pv()) ok = false;
            if (!ok) {
                set_err(p.err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued completes before tensor memory is released
            mma_commit(fin);
            mbar_wait_bounded(fin, 0, p.timeout_ns);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax
        const int r = warp * 32 + lane;                        // query row = TMEM lane
        // bounded wait whose outcome is the same on every lane of the warp
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, p.timeout_ns));
        };
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        const float qnan = __int_as_float(0x7fc00000);
        long long j = 0;
        float m_ref = -INFINITY, l = 0.f;
        int pois = 0, lim = -1;
        bool wact = false, ok = true;
        while (true) {
            if (*abort_flag) break;
            const int st = (int)(j % R);
            if (!wait_all(full(st), (uint32_t)((j / R) & 1))) {
                ok = false;
                break;
            }
            const TcStage rc = recs[st];
            if (rc.flags & TC_END) break;
            if (rc.flags & TC_FIRST) {
                m_ref = -INFINITY;
                l = 0.f;
                pois = 0;
                lim = r < rc.n * G ? rc.ctx - rc.n + r / G : -1;
                wact = __any_sync(0xffffffffu, lim >= 0);
            }
            pois |= rc.poison;
            const int b = (int)(j & 1);
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
                const int kv = min(rc.nkeys, max(0, lim - rc.t0 + 1));    // keys this row sees here
                float mx = -INFINITY;
#pragma unroll
                for (int k = 0; k < KEYS; ++k) {
                    x[k] = k < kv ? x[k] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, x[k]);
                }
                const float m_new = fmaxf(m_ref, mx);
                const bool need = m_new > m_ref + Tr::TAU;
                const float alpha = need ? ex2(m_ref - m_new) : 1.f;      // m_ref = -inf: 0
                if (!(rc.flags & TC_FIRST) && __any_sync(0xffffffffu, need)) {
                    // O holds the earlier stages once their PV is done
                    if (!wait_all(pv_done + 8 * (b ^ 1), (uint32_t)(((j - 1) >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t u[32];
                        tmem_ld32(lane_addr + Tr::O_COL + 32 * c, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
                        tmem_st32(lane_addr + Tr::O_COL + 32 * c, u);
                    }
                    tmem_st_wait();
                }
                if (need) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float mref = m_ref == -INFINITY ? 0.f : m_ref;      // no visible key yet: weights 0
                // P buffer b is free once the PV of stage j - 2 is done
                if (j >= 2 && !wait_all(pv_done + 8 * b, (uint32_t)(((j - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t* prow = smem + Tr::P_OFF + b * 2 * Tr::P_TILE + r * 128;
#pragma unroll
                for (int c = 0; c < KEYS / 8; ++c) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2(x[8 * c + 2 * e] - mref), p1 = ex2(x[8 * c + 2 * e + 1] - mref);
                        l += p0 + p1;
                        const uint32_t h = pack2<Tr::BF16>(p0, p1);
                        hw[e] = h;
                        lw[e] = pack2<Tr::BF16>(p0 - lo_of<Tr::BF16>(h), p1 - hi_of<Tr::BF16>(h));
                    }
                    const int off = (c ^ (r & 7)) << 4;
                    *reinterpret_cast<uint4*>(prow + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(prow + Tr::P_TILE + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            // V rows past the context or past the blocks copied are zero for the PV product
            const int vvalid = max(0, min(rc.nkeys, rc.ctx - rc.t0));
            if (vvalid < KEYS) {
                uint8_t* vt = smem + Tr::RING_OFF + st * Tr::STAGE_BYTES + Tr::KV_BYTES;
                const int nz = (KEYS - vvalid) * HALVES * 8;
                for (int i = threadIdx.x; i < nz; i += 128) {
                    const int row = vvalid + i / (HALVES * 8), part = i % (HALVES * 8);
                    *reinterpret_cast<uint4*>(vt + (part / 8) * Tr::HALF_BYTES + row * 128 + (part % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + 8 * b);
            if (rc.flags & TC_LAST) {
                if (!wait_all(pv_done + 8 * b, (uint32_t)((j >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (wact) {
                    const bool live = lim >= 0;
                    if (rc.flags & TC_COMPLETE) {
                        uint16_t* orow =
                            p.out + ((size_t)(rc.q0 + r / G) * p.Hq + (size_t)rc.kvh * G + r % G) * D;
                        const float inv = 1.f / l;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t u[32];
                            tmem_ld32(lane_addr + Tr::O_COL + 32 * c, u);
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
                                      (((size_t)blockIdx.x * 2 + ((rc.flags & TC_SLOT1) ? 1 : 0)) * Tr::ROWS + r) *
                                          Tr::PSTRIDE;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t u[32];
                            tmem_ld32(lane_addr + Tr::O_COL + 32 * c, u);
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
                            prow[D] = m_ref;
                            prow[D + 1] = l;
                        }
                    }
                }
                tc_fence_before();
            }
            ++j;
        }
        if (!ok) {
            if (lane == 0) set_err(p.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, Tr::TMEM_COLS);
    }
}

template <class Tr>
cudaError_t multi_tc_launch(const MultiLaunch& L) {
    pa_multi_tc_kernel<Tr><<<L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream>>>(*L.tmap_q, *L.tmap_k, *L.tmap_v, L.p);
    return cudaGetLastError();
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
