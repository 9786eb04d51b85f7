// Paged decode attention kernel for sm_103a.
//
// What it computes: for each sequence and query head, softmax attention of the
// newest token's query over the sequence's cached keys/values, which live in
// fixed-size physical blocks reached through a block table (token t sits in
// block table[t / B] at offset t % B -- thewebvale "vLLM & High-Throughput
// Serving", section 2, block-table formula; letsbuildsolutions "How LLM
// Inference Engines Work", PagedAttention section: the kernel must gather K/V
// from non-adjacent memory).  Query heads h of one group share KV head h / g
// (ontq "AI Inference Serving at Scale", section 6, grouped-query attention).
//
// Work split.  The (sequence, KV head) pairs are laid end to end, each
// contributing its blocks; the flattened block list is cut into gridDim.x
// equal contiguous ranges, one per persistent CTA.  A CTA walks its range as
// "segments" (the part of one pair that falls in the range).  A pair that lies
// inside one CTA is finished there; a pair cut by range boundaries leaves a
// partial softmax state (m, l, unnormalised o) per piece in the workspace, and
// the last CTA to finish a piece of that pair (arrival counter, zeroed by the
// host before the launch) merges them with the log-sum-exp rule in CTA order.
// Everything about the split depends on context lengths only, never on block
// ids, so results are bitwise independent of block placement.
//
// Shared prefixes (optional).  With prefix groups, the first first_blocks[s]
// blocks of a member sequence were already reduced by the prefix kernel into
// a per-row state (the carry); here the pair covers only the sequence's own
// blocks after the prefix, and the carry joins the final log-sum-exp
// combination.
//
// Inside a CTA.  Warp NC is the producer: it reads block ids from the table
// (32 at a time, one per lane), and lane 0 issues two-dimensional TMA loads
// (128-byte swizzle) of each (block, KV head) K chunk and V chunk into a ring
// of shared-memory stages guarded by full/empty mbarriers.  Warps 0..NC-1 are
// consumers: block k of the CTA range goes to warp k % NC, which folds it in
// with consume_block() (mma.sync scores, online softmax, PV).  At the end of a
// segment the NC warp states are merged through shared memory.
//
// Every wait is bounded (PA_DEVERR_TIMEOUT); bad block ids and context lengths
// set error bits and poison the affected rows with NaN instead of trapping.
#pragma once

#include <type_traits>

#include "decode_common.cuh"

namespace pa {

struct DecodeParams {
    const uint16_t* q;            // [N][Hq][D]
    const int32_t* block_tables;  // [N][MB]
    const int32_t* context_lens;  // [N]
    uint16_t* out;                // [N][Hq][D]
    int32_t* counters;            // [N * Hkv], zeroed before each launch
    float* partials;              // [gridDim.x][2][G][D + 2]
    uint32_t* err;                // may be null
    // shared prefixes (first_blocks == null: none)
    const int32_t* first_blocks;  // [N] blocks already covered by the prefix pass
    const float* carry;           // [N][Hq][D + 2] prefix states (o, m, l)
    const uint8_t* kv8;           // 8-bit cache only: the pool (K rows, then dims-first V, per piece)
    float v_scale;                // multiplies the output (V's cache scale; 1 for 16-bit)
    int32_t N, Hq, Hkv, NB, MB;
    float scale_log2;             // scale * log2(e)
    uint64_t timeout_ns;
};

// KVF: 0 = the cache holds q's 16-bit type; 1 = FP8 E4M3 codes; 2 = FP8 E5M2.
template <int D_, int BS_, int G_, bool BF16_, int KVF_ = 0>
struct DecodeTraits {
    static constexpr bool KV8 = KVF_ != 0;
    using Gm = std::conditional_t<KV8, Geom8<BS_>, Geom<D_, BS_>>;
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr int UB = Gm::UB;                       // blocks per ring stage
    static constexpr int G = G_;
    static constexpr bool BF16 = BF16_;
    static constexpr bool E5M2 = KVF_ == 2;
    static constexpr int NC = 4;                            // consumer warps
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int MIN_CTAS = 2;
    static constexpr int RING_TARGET = 64 * 1024;
    static constexpr int STAGES =
        ((RING_TARGET / Gm::STAGE_BYTES) > 16 ? 16 : (RING_TARGET / Gm::STAGE_BYTES)) / 4 * 4;
    static constexpr int NR = G > 8 ? 2 : 1;                // 8-row groups of query heads in use
    static constexpr int OSTRIDE = D_ + 4;                  // padded scratch row (bank spread)
    static constexpr int PSTRIDE = D_ + 2;                  // state row: o[D], m, l
    // shared memory carve-up, offsets from a 1024-byte aligned base
    static constexpr int RING_OFF = 0;
    static constexpr int SO_OFF = STAGES * Gm::STAGE_BYTES;
    static constexpr int SO_BYTES = NC * G * OSTRIDE * 4;
    static constexpr int SM_OFF = SO_OFF + SO_BYTES;        // m per (warp, head)
    static constexpr int SL_OFF = SM_OFF + NC * G * 4;      // l per (warp, head)
    static constexpr int SH_OFF = SL_OFF + NC * G * 4;      // per head: M, L, carry factors
    static constexpr int SP_OFF = SH_OFF + 4 * G * 4;       // poison flag per warp
    static constexpr int PS_OFF = SP_OFF + NC * 4;          // poison flag per stage
    static constexpr int BAR_OFF = ((PS_OFF + STAGES * 4) + 7) & ~7;
    static constexpr int INFO_OFF = BAR_OFF + 2 * STAGES * 8;
    static constexpr int INFO_BYTES = 64;
    static constexpr int SMEM_BYTES = INFO_OFF + INFO_BYTES + 1024;  // + alignment slack
    static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "group size");
    static_assert(STAGES >= 2 && STAGES % NC == 0, "ring stages are owned by consumer warps");
};

// Shared CTA bookkeeping written by warp 0 before the roles split.
struct CtaInfo {
    long long lo, hi, W, geff;
    int s0, kvh0, b0;
    int abort;
    int last;
};

// Blocks of sequence s in this kernel's work list (and its first block).
__device__ __forceinline__ int pair_blocks(const DecodeParams& p, int s, int BS, int& first) {
    first = p.first_blocks ? __ldg(p.first_blocks + s) : 0;
    const int nb = seq_blocks(__ldg(p.context_lens + s), BS, p.MB) - first;
    return nb > 0 ? nb : 0;
}

// Position inside the flattened block list, advanced segment by segment.
struct SegIter {
    long long gi;  // flattened index of the next block
    int s, kvh, b0, nb, first;
};

__device__ __forceinline__ void seg_advance(SegIter& it, int len, const DecodeParams& p, int BS) {
    it.gi += len;
    it.b0 += len;
    if (it.b0 == it.nb) {
        it.b0 = 0;
        if (++it.kvh == p.Hkv) {
            it.kvh = 0;
            int nb = 0, first = 0;
            while (++it.s < p.N) {
                nb = pair_blocks(p, it.s, BS, first);
                if (nb > 0) break;
            }
            it.nb = nb;
            it.first = first;
        }
    }
}

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, Tr::MIN_CTAS)
pa_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const DecodeParams p) {
    using Gm = typename Tr::Gm;
    constexpr int D = Tr::D, BS = Tr::BS, G = Tr::G, NC = Tr::NC, S = Tr::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(smem + Tr::RING_OFF);
    float* so = reinterpret_cast<float*>(smem + Tr::SO_OFF);
    float* sm = reinterpret_cast<float*>(smem + Tr::SM_OFF);
    float* sl = reinterpret_cast<float*>(smem + Tr::SL_OFF);
    float* sh = reinterpret_cast<float*>(smem + Tr::SH_OFF);
    int* spois = reinterpret_cast<int*>(smem + Tr::SP_OFF);
    volatile int* stage_poison = reinterpret_cast<volatile int*>(smem + Tr::PS_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::BAR_OFF);
    CtaInfo* info = reinterpret_cast<CtaInfo*>(smem + Tr::INFO_OFF);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, 1);
        }
        fence_mbar_init();
    }
    if constexpr (!Tr::KV8) {
        if (warp == NC && lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
    }

    // ---- work range of this CTA (warp 0) ----
    if (warp == 0) {
        long long w = 0;
        int first = 0;
        for (int s = lane; s < p.N; s += 32) w += pair_blocks(p, s, BS, first);
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        const long long W = w * p.Hkv;
        const long long geff = W < (long long)gridDim.x ? W : (long long)gridDim.x;
        long long lo = 0, hi = 0;
        int s0 = 0, kvh0 = 0, b0 = 0;
        if ((long long)blockIdx.x < geff) {
            lo = range_lo(blockIdx.x, W, geff);
            hi = range_lo(blockIdx.x + 1, W, geff);
            long long base = 0;
            for (int sb = 0; sb < p.N; sb += 32) {
                const int s = sb + lane;
                const long long v = s < p.N ? (long long)pair_blocks(p, s, BS, first) * p.Hkv : 0;
                long long incl = v;
                for (int o = 1; o < 32; o <<= 1) {
                    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const long long total = __shfl_sync(0xffffffffu, incl, 31);
                if (base + total > lo) {
                    const unsigned m = __ballot_sync(0xffffffffu, base + incl > lo);
                    const int firstlane = __ffs(m) - 1;
                    const long long before = base + __shfl_sync(0xffffffffu, incl - v, firstlane);
                    s0 = sb + firstlane;
                    const int nb = pair_blocks(p, s0, BS, first);
                    const long long off = lo - before;
                    kvh0 = (int)(off / nb);
                    b0 = (int)(off % nb);
                    break;
                }
                base += total;
            }
        }
        if (lane == 0) {
            info->lo = lo;
            info->hi = hi;
            info->W = W;
            info->geff = geff;
            info->s0 = s0;
            info->kvh0 = kvh0;
            info->b0 = b0;
            info->abort = 0;
            info->last = 0;
        }
    }

    // ---- rows of sequences with no blocks here: zero (ctx == 0), the prefix
    //      state alone (every key in a shared prefix), NaN (bad ctx) ----
    if (warp < NC) {
        for (int s = blockIdx.x; s < p.N; s += gridDim.x) {
            const int ctx = __ldg(p.context_lens + s);
            int first = 0;
            if (pair_blocks(p, s, BS, first) > 0) continue;
            const bool bad = ctx < 0 || ctx > p.MB * BS;
            if (bad && threadIdx.x == 0) set_err(p.err, PA_DEVERR_CONTEXT);
            uint16_t* row = p.out + (size_t)s * p.Hq * D;
            for (int i = threadIdx.x; i < p.Hq * D; i += NC * 32) {
                uint16_t v = 0;
                if (bad) {
                    v = qnan16<Tr::BF16>();
                } else if (first > 0 && ctx > 0) {
                    const float* c = p.carry + ((size_t)s * p.Hq + i / D) * Tr::PSTRIDE;
                    v = f32_to_16<Tr::BF16>(__ldg(c + i % D) / __ldg(c + D + 1) * p.v_scale);
                }
                row[i] = v;
            }
        }
    }
    __syncthreads();

    const long long lo = info->lo, hi = info->hi, W = info->W, geff = info->geff;
    if ((long long)blockIdx.x >= geff) return;

    SegIter it0;
    it0.gi = lo;
    it0.s = info->s0;
    it0.kvh = info->kvh0;
    it0.b0 = info->b0;
    it0.nb = pair_blocks(p, it0.s, BS, it0.first);

    if (warp == NC) {
        // =========================== producer ===========================
        // One ring stage per UB consecutive blocks of a segment; `issued`
        // counts stages.  A batch of 32 table entries never splits a stage
        // (32 is a multiple of UB).  Stages are filled in rounds: lane j
        // probes (without blocking) whether ring stage issued + j is free,
        // and the leading run of free stages is filled at once, one stage per
        // lane; only when the oldest stage is still busy does lane 0 block on
        // it.  At most S stages are probed per round, so no two lanes touch
        // the same ring slot.
        long long issued = 0;
        bool aborted = false;
        SegIter it = it0;
        while (it.gi < hi && !aborted) {
            const int len = (int)min((long long)(it.nb - it.b0), hi - it.gi);
            const int32_t* trow = p.block_tables + (size_t)it.s * p.MB + it.first + it.b0;
            int tcur = lane < len ? __ldg(trow + lane) : 0;
            for (int base = 0; base < len && !aborted; base += 32) {
                const int nxt = base + 32 + lane < len ? __ldg(trow + base + 32 + lane) : 0;
                const int cnt = min(32, len - base);
                const int nst = (cnt + Tr::UB - 1) / Tr::UB;   // stages in this batch
                int done = 0;
                while (done < nst) {
                    const int want = min(nst - done, S);
                    const long long my = issued + lane;
                    bool is_free = false;
                    if (lane < want)
                        is_free = my < S || mbar_test_wait(empty0 + 8 * (uint32_t)(my % S),
                                                           (uint32_t)(((my / S) - 1) & 1));
                    const unsigned fm = __ballot_sync(0xffffffffu, is_free);
                    int run = (fm == 0xffffffffu) ? 32 : __ffs(~fm) - 1;
                    if (run == 0) {
                        int ok = 1;
                        if (lane == 0)
                            ok = mbar_wait_bounded(empty0 + 8 * (uint32_t)(issued % S),
                                                   (uint32_t)(((issued / S) - 1) & 1), p.timeout_ns) ? 1 : 0;
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) {
                            if (lane == 0) {
                                set_err(p.err, PA_DEVERR_TIMEOUT);
                                *(volatile int*)&info->abort = 1;
                            }
                            aborted = true;
                            break;
                        }
                        run = 1;
                    }
                    // lane j < run fills stage issued + j with batch entries (done + j) * UB ..
                    const int first = (done + lane) * Tr::UB;
                    int ids[Tr::UB];
#pragma unroll
                    for (int u = 0; u < Tr::UB; ++u) ids[u] = __shfl_sync(0xffffffffu, tcur, (first + u) & 31);
                    if (lane < run) {
                        const int nblk = min(Tr::UB, cnt - first);
                        const int st = (int)(my % S);
                        bool bad = false;
#pragma unroll
                        for (int u = 0; u < Tr::UB; ++u) {
                            if (u < nblk && (unsigned)ids[u] >= (unsigned)p.NB) {
                                bad = true;
                                ids[u] = 0;
                            }
                        }
                        if (bad) set_err(p.err, PA_DEVERR_BLOCK_ID);
                        stage_poison[st] = bad ? 1 : 0;
                        const uint32_t fb = full0 + 8 * st;
                        const uint32_t kdst = ring_u32 + st * Gm::STAGE_BYTES;
                        if constexpr (Tr::KV8) {
                            // each block's piece is one contiguous run in the pool
                            mbar_arrive_expect_tx(fb, nblk * Gm::PIECE_BYTES);
#pragma unroll
                            for (int u = 0; u < Tr::UB; ++u)
                                if (u < nblk)
                                    bulk_load(kdst + u * Gm::PIECE_BYTES,
                                              p.kv8 + ((size_t)ids[u] * p.Hkv + it.kvh) * Gm::PIECE_BYTES,
                                              Gm::PIECE_BYTES, fb);
                        } else {
                            mbar_arrive_expect_tx(fb, Gm::STAGE_BYTES);
                            const int y = (ids[0] * p.Hkv + it.kvh) * BS;
#pragma unroll
                            for (int h = 0; h < Gm::HALVES; ++h) {
                                tma_load_2d(kdst + h * Gm::BOX_BYTES, &tmap_k, h * 64, y, fb);
                                tma_load_2d(kdst + Gm::CHUNK_BYTES + h * Gm::BOX_BYTES, &tmap_v, h * 64, y, fb);
                            }
                        }
                    }
                    issued += run;
                    done += run;
                }
                tcur = nxt;
            }
            if (!aborted) seg_advance(it, len, p, BS);
        }
        // Wait until every issued copy has landed before the CTA may exit.
        if (lane == 0) {
            const long long nst = issued < S ? issued : S;
            for (long long st = 0; st < nst; ++st) {
                const long long klast = st + ((issued - 1 - st) / S) * S;
                if (!mbar_wait_bounded(full0 + 8 * (uint32_t)st, (uint32_t)((klast / S) & 1), p.timeout_ns))
                    set_err(p.err, PA_DEVERR_TIMEOUT);
            }
        }
        return;
    }

    // ============================ consumers ============================
    const int tid = threadIdx.x;   // 0 .. NC*32-1
    const int g = lane >> 2;       // fragment row group
    const int t4 = lane & 3;       // fragment column pair
    SegIter it = it0;
    long long ubase = 0;   // stages of the CTA before this segment
    WarpAcc<D, Tr::NR> acc;
    // Q fragments (A operand of S^T = Q K^T), rows = heads of the group
    auto load_q = [&](uint32_t (&qa)[Gm::KD][4], const SegIter& sg) {
        const uint16_t* qrow = p.q + ((size_t)sg.s * p.Hq + (size_t)sg.kvh * G) * D;
        const uint16_t* r0 = g < G ? qrow + g * D : nullptr;
        const uint16_t* r1 = (G > 8) ? qrow + (g + 8) * D : nullptr;
        if constexpr (Tr::KV8) {
            load_q_frags8<D, Tr::BF16>(qa, r0, r1, t4);
        } else {
            load_q_frags<D>(qa, r0, r1, t4);
        }
    };
    uint32_t qa[Gm::KD][4];
    int ctx = 0;
    if (it.gi < hi) {
        ctx = __ldg(p.context_lens + it.s);
        load_q(qa, it);
    }
    while (it.gi < hi) {
        const int len = (int)min((long long)(it.nb - it.b0), hi - it.gi);
        acc.reset();
        int poisoned = 0;

        // Stage k of the CTA (k = ubase + u, UB blocks each) goes to warp
        // k % NC.  With STAGES a multiple of NC every ring stage is owned by one
        // warp, which consumes its fills strictly in order (no mbarrier phase
        // aliasing).
        const int nu = (len + Tr::UB - 1) / Tr::UB;
        int j0 = warp - (int)(ubase % NC);
        if (j0 < 0) j0 += NC;
        for (int u = j0; u < nu; u += NC) {
            const long long k = ubase + u;
            const int st = (int)(k % S);
            const uint32_t par = (uint32_t)((k / S) & 1);
            if (*(volatile int*)&info->abort) {
                poisoned = 1;
                continue;
            }
            if (!mbar_wait_bounded(full0 + 8 * st, par, p.timeout_ns)) {
                if (lane == 0) {
                    set_err(p.err, PA_DEVERR_TIMEOUT);
                    *(volatile int*)&info->abort = 1;
                }
                poisoned = 1;
                continue;
            }
            poisoned |= stage_poison[st];
            const int b = u * Tr::UB;
            const int nblk = min(Tr::UB, len - b);
            const int valid = min(nblk * BS, ctx - (it.first + it.b0 + b) * BS);
            const uint32_t kb = ring_u32 + st * Gm::STAGE_BYTES;
            bool zeroed = false;
            if constexpr (Tr::KV8) {
                if (valid < 32 && (valid & 15)) {
                    zero_v8_tail<Gm>(kb, valid, lane);
                    __syncwarp();
                    zeroed = true;
                }
                consume_stage8<Gm, Tr::NR, Tr::E5M2>(kb, valid, qa, acc, p.scale_log2, lane);
            } else {
                const uint32_t vb = kb + Gm::CHUNK_BYTES;
                if (valid < BS) {
                    zero_v_tail<Gm>(vb, valid, lane);
                    __syncwarp();
                    zeroed = true;
                }
                consume_block<Gm, Tr::NR, Tr::BF16>(kb, vb, valid, qa, acc, p.scale_log2, lane);
            }
            if (zeroed) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
        ubase += nu;

        // The next segment's position, length and Q: loaded now so that the
        // loads overlap the merge below.
        SegIter nx = it;
        seg_advance(nx, len, p, BS);
        int ctx_next = 0;
        if (nx.gi < hi) {
            ctx_next = __ldg(p.context_lens + nx.s);
            load_q(qa, nx);
        }

        // ---- merge the NC warp states of this segment ----
#pragma unroll
        for (int r = 0; r < Tr::NR; ++r) {
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 1);
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 2);
        }
        {
            float* mine = so + warp * G * Tr::OSTRIDE;
#pragma unroll
            for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int head = 8 * r + 2 * t4 + (e & 1);
                        const int dim = 16 * mt + g + 8 * (e >> 1);
                        if (head < G) mine[head * Tr::OSTRIDE + dim] = acc.o[mt][r][e];
                    }
            if (t4 == 0) {
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r) {
                    const int head = g + 8 * r;
                    if (head < G) {
                        sm[warp * G + head] = acc.m[r];
                        sl[warp * G + head] = acc.l[r];
                    }
                }
            }
            if (lane == 0) spois[warp] = poisoned;
        }
        named_bar_sync(1, NC * 32);

        const long long P0 = it.gi - it.b0;           // flattened start of this pair
        const long long cfirst = cta_of(P0, W, geff);
        const long long clast = cta_of(P0 + it.nb - 1, W, geff);
        const bool complete = cfirst == clast;
        const int slot = (it.gi == lo) ? 0 : 1;
        const bool has_carry = it.first > 0;
        int bad = 0;
#pragma unroll
        for (int w = 0; w < NC; ++w) bad |= spois[w];
        const float qnan = __int_as_float(0x7fc00000);
        uint16_t* orow = p.out + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * D;
        const float* crow = p.carry + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * Tr::PSTRIDE;
        float* prow = p.partials + ((size_t)blockIdx.x * 2 + slot) * G * Tr::PSTRIDE;
        // Per head, once: the common max M, each warp's factor exp2(m_w - M)
        // (in place of m_w), L, and for a finished pair with a prefix state
        // the factors that fold the carry in (the log-sum-exp rule).
        if (tid < G) {
            const int hd = tid;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NC; ++w) M = fmaxf(M, sm[w * G + hd]);
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                const float f = ex2(sm[w * G + hd] - M);
                sm[w * G + hd] = f;
                L += sl[w * G + hd] * f;
            }
            float fa = 1.f, fb = 0.f;
            if (complete && has_carry) {
                const float* c = crow + hd * Tr::PSTRIDE;
                const float cm = __ldg(c + D), cl = __ldg(c + D + 1);
                const float Mn = fmaxf(M, cm);
                fa = ex2(M - Mn);
                fb = ex2(cm - Mn);
                L = L * fa + cl * fb;
                M = Mn;
            }
            sh[hd] = M;
            sh[G + hd] = L;
            sh[2 * G + hd] = fa;
            sh[3 * G + hd] = fb;
        }
        named_bar_sync(1, NC * 32);
        for (int idx = tid; idx < G * D; idx += NC * 32) {
            const int head = idx / D;
            const int dim = idx - head * D;
            float O = 0.f;
#pragma unroll
            for (int w = 0; w < NC; ++w) O += so[(w * G + head) * Tr::OSTRIDE + dim] * sm[w * G + head];
            if (bad) O = qnan;
            if (complete) {
                if (has_carry) O = O * sh[2 * G + head] + __ldg(crow + head * Tr::PSTRIDE + dim) * sh[3 * G + head];
                orow[head * D + dim] = f32_to_16<Tr::BF16>(O / sh[G + head] * p.v_scale);
            } else {
                prow[head * Tr::PSTRIDE + dim] = O;
                if (dim == 0) {
                    prow[head * Tr::PSTRIDE + D] = sh[head];
                    prow[head * Tr::PSTRIDE + D + 1] = sh[G + head];
                }
            }
        }

        if (!complete) {
            // Publish this piece, count arrivals; the last piece merges.
            __threadfence();
            named_bar_sync(1, NC * 32);
            const int pair = it.s * p.Hkv + it.kvh;
            if (tid == 0) {
                const int prev = atomicAdd(p.counters + pair, 1);
                *(volatile int*)&info->last = (prev == (int)(clast - cfirst)) ? 1 : 0;
            }
            named_bar_sync(1, NC * 32);
            if (*(volatile int*)&info->last) {
                __threadfence();
                for (int idx = tid; idx < G * D; idx += NC * 32) {
                    const int head = idx / D;
                    const int dim = idx - head * D;
                    float M = -INFINITY, L = 0.f, O = 0.f;
                    for (long long c = cfirst; c <= clast; ++c) {
                        const int sl_c = (c == cfirst && range_lo(c, W, geff) < P0) ? 1 : 0;
                        const float* pr = p.partials + ((size_t)c * 2 + sl_c) * G * Tr::PSTRIDE + head * Tr::PSTRIDE;
                        lse_fold(M, L, O, __ldcg(pr + D), __ldcg(pr + D + 1), __ldcg(pr + dim));
                    }
                    if (has_carry) {
                        const float* cr = crow + head * Tr::PSTRIDE;
                        lse_fold(M, L, O, __ldg(cr + D), __ldg(cr + D + 1), __ldg(cr + dim));
                    }
                    orow[head * D + dim] = f32_to_16<Tr::BF16>(O / L * p.v_scale);
                }
            }
        }
        named_bar_sync(1, NC * 32);
        it = nx;
        ctx = ctx_next;
    }
}

// ---------------------------------------------------------------- host side
struct DecodeLaunch {
    const CUtensorMap* tmap_k;
    const CUtensorMap* tmap_v;
    DecodeParams p;
    cudaStream_t stream;
    int grid;
};

struct DecodeKernelInfo {
    cudaError_t (*launch)(const DecodeLaunch&);
    int (*max_ctas)(int device);   // persistent grid size on that device, <= 0 on error
    int smem_bytes;
    int stages;
};

template <class Tr>
cudaError_t decode_launch(const DecodeLaunch& L) {
    pa_decode_kernel<Tr><<<L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream>>>(*L.tmap_k, *L.tmap_v, L.p);
    return cudaGetLastError();
}

template <class Tr>
DecodeKernelInfo decode_info() {
    return DecodeKernelInfo{&decode_launch<Tr>, &persistent_ctas<pa_decode_kernel<Tr>, Tr::THREADS, Tr::SMEM_BYTES>,
                            Tr::SMEM_BYTES, Tr::STAGES};
}

// Per-(dtype, head_dim) tables, defined in the instantiation units.
// Index: [bs == 32][log2(g)]; the 8-bit tables add [e5m2] in front.
void decode8_table_bf16(DecodeKernelInfo (&t)[2][2][5]);
void decode8_table_fp16(DecodeKernelInfo (&t)[2][2][5]);
void decode_table_bf16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_bf16_d64(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d64(DecodeKernelInfo (&t)[2][5]);

}  // namespace pa
