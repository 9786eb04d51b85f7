// Prefix pass of prefix-aware decode: sequences that share their leading
// physical blocks (parallel samples of one prompt, requests with a common
// system prompt -- ontq "AI Inference Serving at Scale", section 3,
// copy-on-write sharing; letsbuildsolutions, "Production Considerations",
// prefix caching) read those blocks once for the whole group.
//
// Work items are (group, KV head, row chunk): the query rows of a group are
// its members x g query heads of that KV head, taken 32 at a time.  An item
// streams the group's shared blocks (through the first member's table) and
// leaves, for every row, the softmax state (o unnormalised, m, l) of the
// prefix keys in `carry`; the decode kernel then covers each member's own
// blocks and folds the carry in.  Items are cut into equal CTA ranges exactly
// as in the decode kernel, with the same last-arriver merge for items that
// straddle a range boundary.  Every CTA also writes, for the members of each
// well-formed group, how many leading blocks the decode kernel must skip.
//
// Warps: one TMA producer and four consumers arranged as 2 row groups x 2
// block lanes.  Warp (rg, bl) owns rows [16 rg, 16 rg + 16) of the chunk
// (full m16 tiles) and the blocks k of the CTA range with k % 2 == bl; each
// ring stage is read by the two warps of its lane (empty barrier count 2).
// At a segment end the two lanes of each row group merge through shared
// memory.  Shared blocks are full, so no masking is needed.  Each piece also
// checks that every member's table repeats the first member's over the
// prefix and that every member holds at least the prefix; a violation sets
// PA_DEVERR_GROUP and poisons the rows with NaN.
#pragma once

#include "decode_common.cuh"

namespace pa {

struct PrefixParams {
    const uint16_t* q;            // [N][Hq][D]
    const int32_t* block_tables;  // [N][MB]
    const int32_t* context_lens;  // [N]
    const int32_t* grp_starts;    // [n_groups + 1]
    const int32_t* grp_prefix;    // [n_groups]
    float* carry;                 // [N][Hq][D + 2] (o, m, l) out
    int32_t* first_blocks;        // [N] out: prefix blocks of each member (zeroed before the launch)
    int32_t* counters;            // [N * Hkv], zeroed before each launch
    float* partials;              // [gridDim.x][2][32][D + 2]
    uint32_t* err;
    int32_t n_groups, G;          // G: query heads per KV head
    int32_t N, Hq, Hkv, NB, MB;
    float scale_log2;
    uint64_t timeout_ns;
};

template <int D_, int BS_, bool BF16_>
struct PrefixTraits : Geom<D_, BS_> {
    using Gm = Geom<D_, BS_>;
    static constexpr bool BF16 = BF16_;
    static constexpr int NC = 4;                  // consumer warps
    static constexpr int RG = 2;                  // row groups
    static constexpr int BL = NC / RG;            // block lanes
    static constexpr int RPW = 16;                // rows per warp
    static constexpr int RC = RG * RPW;           // rows per item (chunk)
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int STAGES = (64 * 1024 / Gm::STAGE_BYTES) > 16 ? 16 : (64 * 1024 / Gm::STAGE_BYTES);
    static constexpr int PSTRIDE = D_ + 2;
    static constexpr int OSTRIDE = D_ + 4;
    static constexpr int SO_OFF = STAGES * Gm::STAGE_BYTES;
    static constexpr int SM_OFF = SO_OFF + NC * RPW * OSTRIDE * 4;
    static constexpr int SL_OFF = SM_OFF + NC * RPW * 4;
    static constexpr int SP_OFF = SL_OFF + NC * RPW * 4;
    static constexpr int PS_OFF = SP_OFF + NC * 4;
    static constexpr int BAR_OFF = ((PS_OFF + STAGES * 4) + 7) & ~7;
    static constexpr int RF_OFF = BAR_OFF + 2 * STAGES * 8;   // per row: lane factors f0, f1, then M, L
    static constexpr int RP_OFF = RF_OFF + RC * 4 * 4;        // per row: destination row pointer
    static constexpr int MAXP = 8;                            // pieces merged through shared memory
    static constexpr int RSTEP = NC * 32 / (D_ / 2);          // rows apart of one thread's float2 pairs
    static constexpr int EPT = RC / RSTEP;                    // float2 pairs of the row block per thread
    static constexpr int INFO_OFF = RP_OFF + RC * 8;
    static constexpr int INFO_BYTES = 64;
    static constexpr int SMEM_BYTES = INFO_OFF + INFO_BYTES + 1024;
    static_assert(STAGES >= 2 && STAGES % BL == 0, "each ring stage belongs to one block lane");
    static_assert(RC * MAXP <= NC * RPW * OSTRIDE, "piece factors fit in the lane-state area");
    static_assert((NC * 32) % (D_ / 2) == 0 && RC % RSTEP == 0, "the row block splits evenly over the threads");
    static_assert(D_ % 2 == 0 && PSTRIDE % 2 == 0 && OSTRIDE % 2 == 0, "rows hold whole float2 pairs");
};

struct PrefixInfo {
    long long lo, hi, W, geff;
    int g0, kvh0, ch0, b0;
    int abort, last, bad;
};

// Members [s0, s1) and shared blocks of group gi; a malformed description
// yields an empty group and returns false.
__device__ __forceinline__ bool group_of(const PrefixParams& p, int gi, int& s0, int& s1, int& pb) {
    s0 = __ldg(p.grp_starts + gi);
    s1 = __ldg(p.grp_starts + gi + 1);
    pb = __ldg(p.grp_prefix + gi);
    const bool ok = s0 >= 0 && s1 >= s0 && s1 <= p.N && pb >= 0 && pb <= p.MB;
    if (!ok) {
        s0 = s1 = 0;
        pb = 0;
    }
    return ok;
}

__device__ __forceinline__ int group_chunks(const PrefixParams& p, int s0, int s1, int RC) {
    return ((s1 - s0) * p.G + RC - 1) / RC;
}

__device__ __forceinline__ long long group_work(const PrefixParams& p, int gi, int RC) {
    int s0, s1, pb;
    group_of(p, gi, s0, s1, pb);
    return (long long)p.Hkv * group_chunks(p, s0, s1, RC) * pb;
}

struct ItemIter {
    long long gi_flat;   // flattened index of the next block
    int grp, kvh, ch, b0;
    int s0, s1, pb, nch;
};

__device__ __forceinline__ void item_load_group(ItemIter& it, const PrefixParams& p, int RC) {
    while (it.grp < p.n_groups) {
        group_of(p, it.grp, it.s0, it.s1, it.pb);
        it.nch = group_chunks(p, it.s0, it.s1, RC);
        if (it.pb > 0 && it.nch > 0) return;
        ++it.grp;
    }
}

__device__ __forceinline__ void item_advance(ItemIter& it, int len, const PrefixParams& p, int RC) {
    it.gi_flat += len;
    it.b0 += len;
    if (it.b0 == it.pb) {
        it.b0 = 0;
        if (++it.ch == it.nch) {
            it.ch = 0;
            if (++it.kvh == p.Hkv) {
                it.kvh = 0;
                ++it.grp;
                item_load_group(it, p, RC);
            }
        }
    }
}

__device__ __forceinline__ float* carry_row(const PrefixParams& p, int s0, int kvh, int r, int PSTRIDE) {
    return p.carry + ((size_t)(s0 + r / p.G) * p.Hq + (size_t)kvh * p.G + r % p.G) * PSTRIDE;
}

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, 2)
pa_prefix_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const PrefixParams p) {
    using Gm = typename Tr::Gm;
    constexpr int D = Tr::D, BS = Tr::BS, NC = Tr::NC, S = Tr::STAGES, RC = Tr::RC, RG = Tr::RG, BL = Tr::BL;
    constexpr int RPW = Tr::RPW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(smem);
    float* so = reinterpret_cast<float*>(smem + Tr::SO_OFF);
    float* sm = reinterpret_cast<float*>(smem + Tr::SM_OFF);
    float* sl = reinterpret_cast<float*>(smem + Tr::SL_OFF);
    int* spois = reinterpret_cast<int*>(smem + Tr::SP_OFF);
    volatile int* stage_poison = reinterpret_cast<volatile int*>(smem + Tr::PS_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::BAR_OFF);
    PrefixInfo* info = reinterpret_cast<PrefixInfo*>(smem + Tr::INFO_OFF);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, RG);
        }
        fence_mbar_init();
    }
    if (warp == NC && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    // blocks the decode kernel skips for each member of a well-formed group
    for (int gi = blockIdx.x; gi < p.n_groups; gi += gridDim.x) {
        int s0, s1, pb;
        group_of(p, gi, s0, s1, pb);
        for (int s = s0 + threadIdx.x; s < s1; s += Tr::THREADS) p.first_blocks[s] = pb;
    }

    // ---- work range of this CTA (warp 0) ----
    if (warp == 0) {
        long long w = 0;
        bool malformed = false;
        for (int gi = lane; gi < p.n_groups; gi += 32) {
            int s0, s1, pb;
            malformed |= !group_of(p, gi, s0, s1, pb);
            w += (long long)p.Hkv * group_chunks(p, s0, s1, RC) * pb;
        }
        if (__any_sync(0xffffffffu, malformed) && blockIdx.x == 0 && lane == 0) set_err(p.err, PA_DEVERR_GROUP);
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        const long long W = w;
        const long long geff = W < (long long)gridDim.x ? W : (long long)gridDim.x;
        long long lo = 0, hi = 0;
        int g0 = 0, kvh0 = 0, ch0 = 0, b0 = 0;
        if ((long long)blockIdx.x < geff) {
            lo = range_lo(blockIdx.x, W, geff);
            hi = range_lo(blockIdx.x + 1, W, geff);
            long long base = 0;
            for (int gb = 0; gb < p.n_groups; gb += 32) {
                const int gi = gb + lane;
                const long long v = gi < p.n_groups ? group_work(p, gi, RC) : 0;
                long long incl = v;
                for (int o = 1; o < 32; o <<= 1) {
                    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const long long total = __shfl_sync(0xffffffffu, incl, 31);
                if (base + total > lo) {
                    const unsigned m = __ballot_sync(0xffffffffu, base + incl > lo);
                    const int fl = __ffs(m) - 1;
                    const long long before = base + __shfl_sync(0xffffffffu, incl - v, fl);
                    g0 = gb + fl;
                    int s0, s1, pb;
                    group_of(p, g0, s0, s1, pb);
                    const int nch = group_chunks(p, s0, s1, RC);
                    const long long off = lo - before;           // < Hkv * nch * pb
                    const long long item = off / pb;
                    b0 = (int)(off % pb);
                    kvh0 = (int)(item / nch);
                    ch0 = (int)(item % nch);
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
            info->g0 = g0;
            info->kvh0 = kvh0;
            info->ch0 = ch0;
            info->b0 = b0;
            info->abort = 0;
            info->last = 0;
            info->bad = 0;
        }
    }
    __syncthreads();
    const long long lo = info->lo, hi = info->hi, W = info->W, geff = info->geff;
    if ((long long)blockIdx.x >= geff) return;

    ItemIter it0;
    it0.gi_flat = lo;
    it0.grp = info->g0;
    it0.kvh = info->kvh0;
    it0.ch = info->ch0;
    it0.b0 = info->b0;
    group_of(p, it0.grp, it0.s0, it0.s1, it0.pb);
    it0.nch = group_chunks(p, it0.s0, it0.s1, RC);

    if (warp == NC) {
        // =========================== producer ===========================
        // Stages are filled in rounds: lane j probes (without blocking)
        // whether ring stage issued + j is free, and the leading run of free
        // stages is filled at once, one stage per lane; lane 0 blocks only when
        // the oldest stage is still in use.
        long long issued = 0;
        bool aborted = false;
        ItemIter it = it0;
        const uint64_t pol_once = l2_evict_first(), pol_keep = l2_evict_normal();
        while (it.gi_flat < hi && !aborted) {
            const int len = (int)min((long long)(it.pb - it.b0), hi - it.gi_flat);
            const int32_t* trow = p.block_tables + (size_t)it.s0 * p.MB + it.b0;
            int tcur = lane < len ? __ldg(trow + lane) : 0;
            for (int base = 0; base < len && !aborted; base += 32) {
                const int nxt = base + 32 + lane < len ? __ldg(trow + base + 32 + lane) : 0;
                const int cnt = min(32, len - base);
                int done = 0;
                while (done < cnt) {
                    const int want = min(cnt - done, S);
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
                    int id = __shfl_sync(0xffffffffu, tcur, (done + lane) & 31);
                    if (lane < run) {
                        const int st = (int)(my % S);
                        const bool bad = (unsigned)id >= (unsigned)p.NB;
                        if (bad) {
                            set_err(p.err, PA_DEVERR_BLOCK_ID);
                            id = 0;
                        }
                        stage_poison[st] = bad ? 1 : 0;
                        const uint32_t fb = full0 + 8 * st;
                        mbar_arrive_expect_tx(fb, Gm::STAGE_BYTES);
                        const int y = (id * p.Hkv + it.kvh) * BS;
                        const uint32_t kdst = ring_u32 + st * Gm::STAGE_BYTES;
                        // one box per chunk: [column half][BS rows][128 B];
                        // a group of one row chunk reads its blocks once (L2
                        // evict-first), one of several once per chunk
                        const uint64_t pol = it.nch > 1 ? pol_keep : pol_once;
                        tma_load_3d_hint(kdst, &tmap_k, 0, y, 0, fb, pol);
                        tma_load_3d_hint(kdst + Gm::CHUNK_BYTES, &tmap_v, 0, y, 0, fb, pol);
                    }
                    issued += run;
                    done += run;
                }
                tcur = nxt;
            }
            if (!aborted) item_advance(it, len, p, RC);
        }
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
    const int tid = threadIdx.x;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int rg = warp % RG;
    const int bl = warp / RG;
    const float qnan = __int_as_float(0x7fc00000);
    ItemIter it = it0;
    WarpAcc<D, 2> acc;
    while (it.gi_flat < hi) {
        const int len = (int)min((long long)(it.pb - it.b0), hi - it.gi_flat);
        const int R = (it.s1 - it.s0) * p.G;                 // rows of the group for this KV head
        const int rbase = it.ch * RC + rg * RPW;             // first row of this warp
        auto qptr = [&](int r) -> const uint16_t* {
            return r < R ? p.q + ((size_t)(it.s0 + r / p.G) * p.Hq + (size_t)it.kvh * p.G + r % p.G) * D : nullptr;
        };
        uint32_t qa[Gm::KD][4];
        load_q_frags<D>(qa, qptr(rbase + g), qptr(rbase + g + 8), t4);
        acc.reset();
        int poisoned = 0;

        // block k (k = gi_flat - lo) of the range goes to lane k % BL
        int j0 = bl - (int)((it.gi_flat - lo) % BL);
        if (j0 < 0) j0 += BL;
        for (int j = j0; j < len; j += BL) {
            const long long k = it.gi_flat + j - lo;
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
            const uint32_t kb = ring_u32 + st * Gm::STAGE_BYTES;
            consume_block<Gm, 2, Tr::BF16>(kb, kb + Gm::CHUNK_BYTES, BS, qa, acc, p.scale_log2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }

        // ---- the group must really share these blocks ----
        // (a thread per table column; the members' entries are independent loads)
        {
            const int members = it.s1 - it.s0;
            const int32_t* first_row = p.block_tables + (size_t)it.s0 * p.MB;
            int bad = 0;
            for (int m = tid; m < members; m += NC * 32)
                if (__ldg(p.context_lens + it.s0 + m) < it.pb * BS) bad = 1;
            for (int i = tid; i < it.pb; i += NC * 32) {
                const int f = __ldg(first_row + i);
#pragma unroll 4
                for (int m = 1; m < members; ++m)
                    if (__ldg(first_row + (size_t)m * p.MB + i) != f) bad = 1;
            }
            if (bad) atomicOr(&info->bad, 1);
        }

        // ---- write this warp's state; merge the two block lanes ----
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 1);
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 2);
        }
        {
            float* mine = so + warp * RPW * Tr::OSTRIDE;
#pragma unroll
            for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mine[(8 * r + 2 * t4 + (e & 1)) * Tr::OSTRIDE + 16 * mt + g + 8 * (e >> 1)] = acc.o[mt][r][e];
            if (t4 == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    sm[warp * RPW + g + 8 * r] = acc.m[r];
                    sl[warp * RPW + g + 8 * r] = acc.l[r];
                }
            }
            if (lane == 0) spois[warp] = poisoned;
        }
        named_bar_sync(1, NC * 32);
        const bool group_bad = *(volatile int*)&info->bad != 0;
        if (group_bad && tid == 0) set_err(p.err, PA_DEVERR_GROUP);
        int anybad = group_bad ? 1 : 0;
#pragma unroll
        for (int w = 0; w < NC; ++w) anybad |= spois[w];

        const long long P0 = it.gi_flat - it.b0;
        const long long cfirst = cta_of(P0, W, geff);
        const long long clast = cta_of(P0 + it.pb - 1, W, geff);
        const bool complete = cfirst == clast;
        const int slot = (it.gi_flat == lo) ? 0 : 1;
        const int rows = min(RC, R - it.ch * RC);
        float* prow = p.partials + ((size_t)blockIdx.x * 2 + slot) * RC * Tr::PSTRIDE;
        // per row, once: the factors that merge the two block lanes of its
        // row group, the merged m and l, and where the row goes
        float* rowf = reinterpret_cast<float*>(smem + Tr::RF_OFF);
        float** rowp = reinterpret_cast<float**>(smem + Tr::RP_OFF);
        if (tid < rows) {
            const int rr = tid % RPW;
            const int w0 = tid / RPW, w1 = w0 + RG;           // the two lanes of this row group
            const float m0 = sm[w0 * RPW + rr], m1 = sm[w1 * RPW + rr];
            const float M = fmaxf(m0, m1);
            const float f0 = ex2(m0 - M), f1 = ex2(m1 - M);
            float* dst = complete ? carry_row(p, it.s0, it.kvh, it.ch * RC + tid, Tr::PSTRIDE)
                                  : prow + tid * Tr::PSTRIDE;
            rowf[4 * tid] = f0;
            rowf[4 * tid + 1] = f1;
            dst[D] = M;
            dst[D + 1] = sl[w0 * RPW + rr] * f0 + sl[w1 * RPW + rr] * f1;
            rowp[tid] = dst;
        }
        named_bar_sync(1, NC * 32);
        // o of every row: thread tid owns dims c2, c2 + 1 of rows tid / (D / 2) + j * RSTEP,
        // all read before any is written
        const int c2 = 2 * (tid % (D / 2));
        {
            float2 o[Tr::EPT];
#pragma unroll
            for (int j = 0; j < Tr::EPT; ++j) {
                const int rloc = tid / (D / 2) + j * Tr::RSTEP;
                const int rr = rloc % RPW;
                const int w0 = rloc / RPW, w1 = w0 + RG;
                const float f0 = rowf[4 * rloc], f1 = rowf[4 * rloc + 1];
                const float2 a = *reinterpret_cast<const float2*>(so + (w0 * RPW + rr) * Tr::OSTRIDE + c2);
                const float2 b = *reinterpret_cast<const float2*>(so + (w1 * RPW + rr) * Tr::OSTRIDE + c2);
                o[j] = anybad ? make_float2(qnan, qnan) : make_float2(a.x * f0 + b.x * f1, a.y * f0 + b.y * f1);
            }
#pragma unroll
            for (int j = 0; j < Tr::EPT; ++j) {
                const int rloc = tid / (D / 2) + j * Tr::RSTEP;
                if (rloc < rows) *reinterpret_cast<float2*>(rowp[rloc] + c2) = o[j];
            }
        }

        if (!complete) {
            __threadfence();
            named_bar_sync(1, NC * 32);
            const int cid = (it.s0 + it.ch * (RC / p.G)) * p.Hkv + it.kvh;
            if (tid == 0) {
                const int prev = atomicAdd(p.counters + cid, 1);
                *(volatile int*)&info->last = (prev == (int)(clast - cfirst)) ? 1 : 0;
            }
            named_bar_sync(1, NC * 32);
            const int np = (int)(clast - cfirst + 1);
            if (*(volatile int*)&info->last && np <= Tr::MAXP) {
                // the item's pieces, in CTA order; the first CTA's piece is in
                // its second slot when its range starts inside the item
                __threadfence();
                const int sl0 = range_lo(cfirst, W, geff) < P0 ? 1 : 0;
                auto piece = [&](int k) -> const float* {
                    return p.partials + ((size_t)(cfirst + k) * 2 + (k == 0 ? sl0 : 0)) * RC * Tr::PSTRIDE;
                };
                float* fct = so;                               // [RC][MAXP], the lane states are consumed
                if (tid < rows) {
                    float mk[Tr::MAXP];
                    float M = -INFINITY;
#pragma unroll
                    for (int k = 0; k < Tr::MAXP; ++k) {
                        mk[k] = k < np ? __ldcg(piece(k) + tid * Tr::PSTRIDE + D) : -INFINITY;
                        M = fmaxf(M, mk[k]);
                    }
                    float L = 0.f;
#pragma unroll
                    for (int k = 0; k < Tr::MAXP; ++k) {
                        if (k < np) {
                            const float f = ex2(mk[k] - M);
                            L += __ldcg(piece(k) + tid * Tr::PSTRIDE + D + 1) * f;
                            fct[tid * Tr::MAXP + k] = f;
                        }
                    }
                    float* dst = carry_row(p, it.s0, it.kvh, it.ch * RC + tid, Tr::PSTRIDE);
                    dst[D] = M;
                    dst[D + 1] = L;
                    rowp[tid] = dst;
                }
                named_bar_sync(1, NC * 32);
                // piece by piece, each thread's rows at once (loads of one
                // piece are independent), then the writes
                float2 o[Tr::EPT];
#pragma unroll
                for (int j = 0; j < Tr::EPT; ++j) o[j] = make_float2(0.f, 0.f);
                for (int k = 0; k < np; ++k) {
                    const float* pk = piece(k);
#pragma unroll
                    for (int j = 0; j < Tr::EPT; ++j) {
                        const int rloc = tid / (D / 2) + j * Tr::RSTEP;
                        if (rloc < rows) {
                            const float f = fct[rloc * Tr::MAXP + k];
                            const float2 v = __ldcg(reinterpret_cast<const float2*>(pk + rloc * Tr::PSTRIDE + c2));
                            o[j].x += v.x * f;
                            o[j].y += v.y * f;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < Tr::EPT; ++j) {
                    const int rloc = tid / (D / 2) + j * Tr::RSTEP;
                    if (rloc < rows) *reinterpret_cast<float2*>(rowp[rloc] + c2) = o[j];
                }
            } else if (*(volatile int*)&info->last) {
                // more pieces than the shared-memory path holds: fold them in
                // order, element by element
                __threadfence();
                for (int idx = tid; idx < rows * (D + 2); idx += NC * 32) {
                    const int rloc = idx / (D + 2);
                    const int col = idx - rloc * (D + 2);
                    float M = -INFINITY, L = 0.f, O = 0.f;
                    for (long long c = cfirst; c <= clast; ++c) {
                        const int sl_c = (c == cfirst && range_lo(c, W, geff) < P0) ? 1 : 0;
                        const float* pr = p.partials + ((size_t)c * 2 + sl_c) * RC * Tr::PSTRIDE + rloc * Tr::PSTRIDE;
                        lse_fold(M, L, O, __ldcg(pr + D), __ldcg(pr + D + 1), col < D ? __ldcg(pr + col) : 0.f);
                    }
                    float* dst = carry_row(p, it.s0, it.kvh, it.ch * RC + rloc, Tr::PSTRIDE);
                    dst[col] = col < D ? O : (col == D ? M : L);
                }
            }
        }
        named_bar_sync(1, NC * 32);
        if (tid == 0) info->bad = 0;
        named_bar_sync(1, NC * 32);
        item_advance(it, len, p, RC);
    }
}

struct PrefixLaunch {
    const CUtensorMap* tmap_k;
    const CUtensorMap* tmap_v;
    PrefixParams p;
    cudaStream_t stream;
    int grid;
};

struct PrefixKernelInfo {
    cudaError_t (*launch)(const PrefixLaunch&);
    int (*max_ctas)(int device);
};

template <class Tr>
cudaError_t prefix_launch(const PrefixLaunch& L) {
    pa_prefix_kernel<Tr><<<L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream>>>(*L.tmap_k, *L.tmap_v, L.p);
    return cudaGetLastError();
}

template <class Tr>
PrefixKernelInfo prefix_info() {
    return PrefixKernelInfo{&prefix_launch<Tr>, &persistent_ctas<pa_prefix_kernel<Tr>, Tr::THREADS, Tr::SMEM_BYTES>};
}

// Index: [bf16][d == 128][bs == 32]; defined in prefix_inst.cu.
void prefix_table(PrefixKernelInfo (&t)[2][2][2]);

}  // namespace pa
