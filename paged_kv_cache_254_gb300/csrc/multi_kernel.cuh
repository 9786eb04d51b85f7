// Paged attention for a chunk of query tokens per sequence (chunked prefill,
// speculative verification) on sm_103a.
//
// What it computes: sequence s brings q_len = q_start[s + 1] - q_start[s]
// query tokens, its last q_len cached tokens (their K/V were appended before
// the call); query token i attends causally to the keys t <= ctx - q_len + i,
// gathered through the block table (thewebvale "vLLM & High-Throughput
// Serving", section 4, chunked prefill; letsbuildsolutions "How LLM Inference
// Engines Work", speculative decoding: the target model checks every drafted
// token in one pass).  Query heads h of one group share KV head h / g.
//
// Rows.  For a (sequence, KV head) pair the query rows are r = i * g + hh
// (token i of the chunk, head hh of the group): q_len * g <= 16 * NW rows,
// 16 per warp (one m16 tile of the score MMA, as in the decode kernel).  The
// library runs this kernel with NW = 1 (launches of up to 16 rows per pair);
// larger ones go to the tcgen05 kernel (multi_tc_kernel.cuh), whose 128-row
// tile costs the same at any row count.
//
// Work split.  The pairs' blocks are laid end to end and cut into one equal
// contiguous chunk per CTA (the decode kernel's static split).  A CTA reads
// each block of its chunk once into a ring of R stages that all its NW warps
// read: a full mbarrier per stage (the copy landed) and an empty mbarrier
// counting the warps that are done with it.  Lane 0 of warp 0 issues the
// copies R stages ahead, refilling a stage once every warp has released it.
// A pair cut by chunk boundaries leaves per-row partial states; the merge
// post-pass combines them in chunk order.
//
// Masking.  Scores of keys past a row's limit are -inf (per row: the two rows
// a lane holds have their own limits).  The running max starts at -inf and a
// row can meet a stage with no visible key, so exponentials are taken against
// 0 while the max is still -inf.  K/V slots past the context may hold anything
// (NaN included): masked scores never use K, and the V entries of those slots
// are zeroed in the MMA operand registers, so the shared stage is never
// written and all warps can read it.
//
// Every wait is bounded; bad data sets error bits and poisons rows with NaN.
#pragma once

#include "decode_kernel.cuh"

namespace pa {

template <int D_, int BS_, int NW_, bool BF16_>
struct MultiTraits {
    using Gm = Geom<D_, BS_>;
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr int NW = NW_;                          // warps = 16-row tiles per CTA
    static constexpr int ROWS = 16 * NW;
    static constexpr bool BF16 = BF16_;
    static constexpr int THREADS = 32 * NW;
    // about 8 warps per SM: 6 / 4 / 2 / 1 CTAs of 1 / 2 / 4 / 8 warps, sharing
    // ~190 KiB of stages
    static constexpr int MIN_CTAS = NW == 1 ? 6 : NW == 2 ? 4 : NW == 4 ? 2 : 1;
    static constexpr int RING = (NW == 8 ? 192 : 160) * 1024 / MIN_CTAS;
    static constexpr int R_FIT = RING / Gm::STAGE_BYTES;
    static constexpr int R = R_FIT > 24 ? 24 : (R_FIT < 2 ? 2 : R_FIT);   // ring stages of the CTA
    static constexpr int PSTRIDE = D_ + 4;                  // partial row: o[D], m, l, 2 pad
    static constexpr int CUM_SMEM = 256;
    static constexpr int BAR_OFF = R * Gm::STAGE_BYTES;
    static constexpr int CUM_OFF = BAR_OFF + 2 * R * 8;
    static constexpr int CTX_OFF = CUM_OFF + (CUM_SMEM + 1) * 8;
    static constexpr int QS_OFF = CTX_OFF + CUM_SMEM * 4;
    static constexpr int PS_OFF = QS_OFF + (CUM_SMEM + 1) * 4;
    static constexpr int AB_OFF = PS_OFF + R * 4;
    static constexpr int SMEM_BYTES = AB_OFF + 16 + 1024;  // + alignment slack
    static_assert(R >= 2, "ring");
    static_assert(NW == 1 || NW == 2 || NW == 4 || NW == 8, "warps");
};

// consume_block for query rows with their own key limits: valid[r] keys of
// this block are visible to the lane's row group r (rows g and g + 8 of the
// warp's tile), vvalid slots of the block hold cached tokens (the rest of the
// V rows are zeroed in registers).
template <class Gm, bool BF16>
__device__ __forceinline__ void consume_block_rows(uint32_t kb, uint32_t vb, const int (&valid)[2], int vvalid,
                                                   const uint32_t (&qa)[Gm::KD][4], WarpAcc<Gm::D, 2>& acc,
                                                   float scale_log2, int lane) {
    constexpr int NR = 2;
    const int t4 = lane & 3;
    float sacc[Gm::NT][4];
#pragma unroll
    for (int nt = 0; nt < Gm::NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < Gm::KD / 2; ++q4) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + swz<Gm::BOX_BYTES>(nt * 8 + (lane & 7), q4 * 4 + (lane >> 3)), b0, b1, b2, b3);
            mma16816<BF16>(sacc[nt], qa[2 * q4][0], qa[2 * q4][1], qa[2 * q4][2], qa[2 * q4][3], b0, b1);
            mma16816<BF16>(sacc[nt], qa[2 * q4 + 1][0], qa[2 * q4 + 1][1], qa[2 * q4 + 1][2], qa[2 * q4 + 1][3],
                           b2, b3);
        }
    }
    float mx[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) mx[r] = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + 2 * t4 + (e & 1);
            const float v = tok < valid[e >> 1] ? sacc[nt][e] * scale_log2 : -INFINITY;
            sacc[nt][e] = v;
            mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
    float alpha[NR], mref[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(acc.m[r], mx[r]);
        mref[r] = m_new == -INFINITY ? 0.f : m_new;          // no visible key yet: exponentials give 0
        alpha[r] = ex2(acc.m[r] - mref[r]);
        acc.m[r] = m_new;
        acc.l[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = e >> 1;
            const float pe = ex2(sacc[nt][e] - mref[r]);
            sacc[nt][e] = pe;
            acc.l[r] += pe;
        }
    uint32_t pb[Gm::KT][NR][2], pl[Gm::KT][NR][2];
#pragma unroll
    for (int kt = 0; kt < Gm::KT; ++kt)
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float x0 = sacc[2 * kt + h][2 * r], x1 = sacc[2 * kt + h][2 * r + 1];
                const uint32_t hi = pack2<BF16>(x0, x1);
                pb[kt][r][h] = hi;
                pl[kt][r][h] = pack2<BF16>(x0 - lo_of<BF16>(hi), x1 - hi_of<BF16>(hi));
            }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float aa = __shfl_sync(0xffffffffu, alpha[r], (2 * t4) * 4);
        const float ab = __shfl_sync(0xffffffffu, alpha[r], (2 * t4 + 1) * 4);
#pragma unroll
        for (int mt = 0; mt < Gm::KD; ++mt) {
            acc.o[mt][r][0] *= aa;
            acc.o[mt][r][1] *= ab;
            acc.o[mt][r][2] *= aa;
            acc.o[mt][r][3] *= ab;
        }
    }
    // V^T operand registers: a0 / a1 hold the tokens 16 kt + 2 t4 + {0, 1},
    // a2 / a3 the tokens 16 kt + 8 + 2 t4 + {0, 1} (low half = the first)
    auto keep = [&](int tok) -> uint32_t {
        return (tok < vvalid ? 0x0000ffffu : 0u) | (tok + 1 < vvalid ? 0xffff0000u : 0u);
    };
#pragma unroll
    for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
        for (int kt = 0; kt < Gm::KT; ++kt) {
            uint32_t a0, a1, a2, a3;
            const int row = kt * 16 + ((lane >> 4) << 3) + (lane & 7);
            const int chunk = 2 * mt + ((lane >> 3) & 1);
            ldsm_x4_t(vb + swz<Gm::BOX_BYTES>(row, chunk), a0, a1, a2, a3);
            if (vvalid < Gm::BS) {
                const uint32_t k0 = keep(16 * kt + 2 * t4), k1 = keep(16 * kt + 8 + 2 * t4);
                a0 &= k0;
                a1 &= k0;
                a2 &= k1;
                a3 &= k1;
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                mma16816<BF16>(acc.o[mt][r], a0, a1, a2, a3, pb[kt][r][0], pb[kt][r][1]);
                mma16816<BF16>(acc.o[mt][r], a0, a1, a2, a3, pl[kt][r][0], pl[kt][r][1]);
            }
        }
}

struct MultiParams {
    DecodeParams d;               // q / out hold T = q_start[N] token rows
    const int32_t* q_start;       // [N + 1] first query row of each sequence
    int32_t max_q;                // the launch's largest chunk (q_len above it is an error)
    int32_t total_q;              // T: rows of q and out
    int32_t q_box;                // tokens per Q tile copy (tensor-core kernel: min(max_q, T))
};

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, Tr::MIN_CTAS)
pa_multi_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                const MultiParams mp) {
    using Gm = typename Tr::Gm;
    constexpr int D = Tr::D, BS = Tr::BS, NW = Tr::NW, R = Tr::R, ROWS = Tr::ROWS;
    const DecodeParams& p = mp.d;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int G = p.Hq / p.Hkv;
    const uint32_t ring = smem_u32(smem);
    const uint32_t full0 = smem_u32(smem + Tr::BAR_OFF);
    const uint32_t empty0 = full0 + R * 8;
    volatile int* stage_poison = reinterpret_cast<volatile int*>(smem + Tr::PS_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Tr::AB_OFF);
    long long* scum = reinterpret_cast<long long*>(smem + Tr::CUM_OFF);
    int* sctx = reinterpret_cast<int*>(smem + Tr::CTX_OFF);
    int* sqs = reinterpret_cast<int*>(smem + Tr::QS_OFF);

    if (threadIdx.x == 0) {
        for (int st = 0; st < R; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, NW);
        }
        fence_mbar_init();
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        *abort_flag = 0;
    }
    // launched with programmatic stream serialization after the pre-pass:
    // the set-up above overlaps it; nothing the stream wrote is read before
    // it completes.  The merge post-pass may then be placed as CTAs retire.
    griddep_wait();
    griddep_launch_dependents();
    const bool in_smem = p.N <= Tr::CUM_SMEM;
    if (in_smem) {
        for (int i = threadIdx.x; i <= p.N; i += Tr::THREADS) {
            scum[i] = __ldg(p.cum + i);
            sqs[i] = __ldg(mp.q_start + i);
            if (i < p.N) sctx[i] = __ldg(p.context_lens + i);
        }
    }
    __syncthreads();
    SeqTab tab;
    tab.cum = in_smem ? scum : p.cum;
    tab.ctx = in_smem ? sctx : p.context_lens;
    tab.first = nullptr;
    const int* qst = in_smem ? sqs : mp.q_start;
    const long long* cum = tab.cum;
    const float qnan = __int_as_float(0x7fc00000);
    // a sequence's chunk length, or -1 when it is malformed
    auto chunk_len = [&](int s) -> int {
        const int a = qst[s], b = qst[s + 1], ctx = tab.ctx[s];
        const int n = b - a;
        const bool ok = a >= 0 && b <= mp.total_q && n >= 0 && n <= mp.max_q && n <= (ctx > 0 ? ctx : 0);
        return ok ? n : -1;
    };

    // ---- sequences with no blocks (ctx == 0: an empty chunk is all there can
    //      be; bad ctx) and malformed chunks: error bit, NaN rows where the
    //      rows can be named ----
    for (int s = blockIdx.x; s < p.N; s += gridDim.x) {
        const int n = chunk_len(s);
        const int ctx = tab.ctx[s];
        const bool bad_ctx = ctx < 0 || ctx > p.MB * BS;
        if (n >= 0 && !bad_ctx) continue;
        if (threadIdx.x == 0) set_err(p.err, PA_DEVERR_CONTEXT);
        const int a = max(0, qst[s]);
        const int b = min(mp.total_q, qst[s + 1]);
        for (long long i = (long long)a * p.Hq * D + threadIdx.x; i < (long long)b * p.Hq * D; i += Tr::THREADS)
            p.out[i] = qnan16<Tr::BF16>();
    }

    // ---- this CTA's chunk ----
    const Sched sc = make_sched(cum[p.N] * p.Hkv, gridDim.x, 0);
    if ((int)blockIdx.x >= sc.NS) return;
    const long long lo = sc.lo(blockIdx.x), hi = sc.lo(blockIdx.x + 1);
    SegIter it = locate(p, tab, lo, lane);

    // ---- issue side (lane 0 of warp 0) ----
    SegIter is = it;
    int ilen = seg_len(is, hi), ib = 0, tbase = 0;
    const int32_t* irow = p.block_tables + (size_t)is.s * p.MB + is.b0;
    auto row_ids = [&](const int32_t* row, int off, int navail) -> int {
        return lane < navail ? __ldg(row + off + lane) : 0;
    };
    int tcur = 0, tnxt = 0;
    if (warp == 0) {
        tcur = row_ids(irow, 0, ilen);
        tnxt = row_ids(irow, 32, ilen - 32);
    }
    long long nis = 0;
    int ist = 0;               // nis % R, kept without a division
    bool idone = false;
    const uint64_t kv_pol = l2_evict_first();
    auto issue_one = [&]() {   // warp 0 only; the stage's slot is known to be free
        if (idone) return;
        const int st = ist;
        if (++ist == R) ist = 0;
        int id = __shfl_sync(0xffffffffu, tcur, (ib - tbase) & 31);
        const bool bad = (unsigned)id >= (unsigned)p.NB;
        if (bad) id = 0;
        const uint32_t fb = full0 + 8 * st;
        if (lane == 0) {
            if (bad) set_err(p.err, PA_DEVERR_BLOCK_ID);
            stage_poison[st] = bad ? 1 : 0;
            mbar_arrive_expect_tx(fb, Gm::STAGE_BYTES);
        }
        __syncwarp();
        // one box per chunk ([column half][BS rows][128 B]): K from lane 0, V
        // from lane 1, side by side
        // (read once: L2 evict-first)
        if (lane < 2)
            tma_load_3d_hint(ring + st * Gm::STAGE_BYTES + (lane ? Gm::CHUNK_BYTES : 0), lane ? &tmap_v : &tmap_k,
                             0, (id * p.Hkv + is.kvh) * BS, 0, fb, kv_pol);
        ++nis;
        ++ib;
        if (ib == ilen) {
            seg_advance(is, ilen, p, tab);
            if (is.gi < hi) {
                ilen = seg_len(is, hi);
                ib = 0;
                tbase = 0;
                irow = p.block_tables + (size_t)is.s * p.MB + is.b0;
                tcur = row_ids(irow, 0, ilen);
                tnxt = row_ids(irow, 32, ilen - 32);
            } else {
                idone = true;
            }
        } else if (ib - tbase == 32) {
            tbase += 32;
            tcur = tnxt;
            tnxt = row_ids(irow, tbase + 32, ilen - tbase - 32);
        }
    };
    if (warp == 0)
        for (int i = 0; i < R; ++i) issue_one();

    // ---- every warp: its 16 rows of each pair ----
    const int rw0 = warp * 16 + g, rw1 = rw0 + 8;   // tile rows this lane holds (row groups 0, 1)
    auto load_q = [&](uint32_t (&qa)[Gm::KD][4], const SegIter& sg, int n) {
        const int base = n > 0 ? qst[sg.s] : 0;
        auto row = [&](int rr) -> const uint16_t* {
            if (rr >= n * G) return nullptr;
            return p.q + ((size_t)(base + rr / G) * p.Hq + (size_t)sg.kvh * G + rr % G) * D;
        };
        load_q_frags<D>(qa, row(rw0), row(rw1), t4);
    };
    WarpAcc<D, 2> acc;
    uint32_t qa[Gm::KD][4];
    int nq = max(0, chunk_len(it.s));
    load_q(qa, it, nq);
    long long ncons = 0;
    int cst = 0;               // ncons % R
    uint32_t cph = 0;          // (ncons / R) & 1
    while (it.gi < hi) {
        const int len = seg_len(it, hi);
        const int ctx = tab.ctx[it.s];
        const int n_raw = chunk_len(it.s);
        const bool seq_bad = n_raw < 0;
        const int n = max(0, n_raw);
        SegIter nx = it;
        seg_advance(nx, len, p, tab);
        const bool nx_here = nx.gi < hi;
        uint32_t qn[Gm::KD][4];
        int n_next = 0;
        if (nx_here) {
            n_next = max(0, chunk_len(nx.s));
            load_q(qn, nx, n_next);
        }
        // key limits of the lane's two rows (-1: no such row)
        const int lim0 = rw0 < n * G ? ctx - n + rw0 / G : -1;
        const int lim1 = rw1 < n * G ? ctx - n + rw1 / G : -1;
        acc.reset();
        int poisoned = seq_bad ? 1 : 0;
        for (int b = 0; b < len; ++b) {
            const int st = cst;
            const uint32_t par = cph;
            if (++cst == R) {
                cst = 0;
                cph ^= 1u;
            }
            ++ncons;
            if (*abort_flag) {
                poisoned = 1;
                continue;
            }
            if (!mbar_wait_bounded(full0 + 8 * st, par, p.timeout_ns)) {
                if (lane == 0) {
                    set_err(p.err, PA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                poisoned = 1;
                continue;
            }
            poisoned |= stage_poison[st];
            const int t0 = (it.b0 + b) * BS;
            const int valid[2] = {min(BS, max(0, lim0 - t0 + 1)), min(BS, max(0, lim1 - t0 + 1))};
            const int vvalid = min(BS, ctx - t0);
            const uint32_t kb = ring + st * Gm::STAGE_BYTES;
            consume_block_rows<Gm, Tr::BF16>(kb, kb + Gm::CHUNK_BYTES, valid, vvalid, qa, acc, p.scale_log2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            if (warp == 0 && !idone) {
                // refill this slot once every warp has released it
                const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * st, par, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) {
                        set_err(p.err, PA_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    idone = true;
                } else {
                    issue_one();
                }
            }
        }

        // ---- finish the segment: this warp's rows ----
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 1);
            acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 2);
        }
        const long long P0 = it.gi - it.b0;
        const long long cfirst = sc.of(P0), clast = sc.of(P0 + it.nb - 1);
        const bool complete = cfirst == clast;
        const int slot = (it.gi == lo) ? 0 : 1;
        float* prow = p.partials + ((size_t)blockIdx.x * 2 + slot) * ROWS * Tr::PSTRIDE;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                // this lane's o columns are tile rows warp*16 + 8 r + 2 t4 + c
                const int rr = warp * 16 + 8 * r + 2 * t4 + c;
                const float L = __shfl_sync(0xffffffffu, acc.l[r], (2 * t4 + c) * 4);
                if (rr < n * G) {
                    if (complete) {
                        uint16_t* orow = p.out + ((size_t)(qst[it.s] + rr / G) * p.Hq + (size_t)it.kvh * G + rr % G) * D;
                        const float inv = 1.f / L;
#pragma unroll
                        for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const float O = poisoned ? qnan : acc.o[mt][r][2 * hh + c];
                                orow[16 * mt + g + 8 * hh] = f32_to_16<Tr::BF16>(O * inv);
                            }
                    } else {
#pragma unroll
                        for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                prow[rr * Tr::PSTRIDE + 16 * mt + g + 8 * hh] = poisoned ? qnan : acc.o[mt][r][2 * hh + c];
                    }
                }
            }
        if (!complete && t4 == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rr = warp * 16 + g + 8 * r;
                if (rr < n * G) {
                    prow[rr * Tr::PSTRIDE + D] = acc.m[r];
                    prow[rr * Tr::PSTRIDE + D + 1] = acc.l[r];
                }
            }
        }
        if (!nx_here) break;
        it = nx;
#pragma unroll
        for (int kk = 0; kk < Gm::KD; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i) qa[kk][i] = qn[kk][i];
        (void)n_next;
    }

    // After an abort, wait (bounded) for the copies still in flight before the
    // CTA's shared memory is released.
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (long long k = nis - R > 0 ? nis - R : 0; k < nis; ++k)
            mbar_wait_bounded(full0 + 8 * (uint32_t)(k % R), (uint32_t)((k / R) & 1), p.timeout_ns);
    }
}

// Post-pass: rows of pairs cut by chunk boundaries, combined in chunk order
// by the log-sum-exp rule.  A pair is cut where a chunk boundary falls
// strictly inside it; one CTA per boundary, and the first boundary inside a
// pair merges it (the others return), so only cut pairs cost work.  Each warp
// merges rows of the pair: D / 4 lanes per row, 4 dims each.  With up to
// MERGE_PIECES pieces, a row's (m, l, o slice) of every piece are loaded in
// one round before any is used (one memory latency per row, and the CTA's
// MERGE_THREADS / 32 warps keep that many rows in flight); more pieces take
// two passes.
constexpr int MERGE_THREADS = 512;
constexpr int MERGE_PIECES = 4;

template <int D>
__global__ void __launch_bounds__(MERGE_THREADS)
pa_multi_merge(const long long* __restrict__ cum, const int32_t* __restrict__ q_start,
               const int32_t* __restrict__ context_lens, const float* __restrict__ partials,
               uint16_t* __restrict__ out, int N, int Hkv, int G, int rows_per_chunk, int nchunks_hint,
               int max_q, int total_q, int bf16) {
    griddep_wait();   // the attention grid is complete and its writes visible
    constexpr int PSTRIDE = D + 4;
    constexpr int LPR = D / 4;                    // lanes per row
    constexpr int RPW = 32 / LPR;                 // rows per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int sub = lane % LPR;
    const long long W = cum[N] * Hkv;
    const Sched sc = make_sched(W, nchunks_hint, 0);
    const int c = (int)blockIdx.x + 1;            // boundary between chunks c - 1 and c
    if (c >= sc.NS) return;
    const long long x = sc.lo(c);
    // the pair holding flattened block x: sequence s with cum[s] Hkv <= x <
    // cum[s + 1] Hkv, by a 32-way search (one probe per lane per round, so
    // two rounds of dependent loads up to 1,024 sequences); every warp runs
    // it, so the block needs no barrier
    int a = 0, b = N;
    while (b - a > 1) {
        const int step = (b - a + 31) / 32;
        const int idx = a + lane * step;
        const bool le = idx < b && cum[idx] * Hkv <= x;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        a += (31 - __clz(m)) * step;                  // lane 0 probes a, which always holds
        b = min(a + step, b);
    }
    const int s = a;
    const int nb = (int)(cum[s + 1] - cum[s]);
    if (nb == 0) return;
    const int kvh = (int)((x - cum[s] * Hkv) / nb);
    const long long P0 = cum[s] * Hkv + (long long)kvh * nb;
    if (P0 == x || sc.lo(c - 1) > P0) return;     // not cut here, or cut first by an earlier boundary
    const int qa = q_start[s], qb = q_start[s + 1];
    const int n = qb - qa;
    const int ctx = context_lens[s];
    if (qa < 0 || qb > total_q || n < 0 || n > max_q || n > ctx) return;    // reported by the kernel
    const long long cfirst = sc.of(P0), clast = sc.of(P0 + nb - 1);
    const size_t cstride = (size_t)2 * rows_per_chunk * PSTRIDE;
    const int np = (int)(clast - cfirst) + 1;
    const int d0 = sub * 4;
    const int Hq = Hkv * G;
    for (int base = warp * RPW; base < n * G; base += nwarps * RPW) {
        const int rr = base + lane / LPR;
        const bool writer = rr < n * G;
        const int row = writer ? rr : 0;
        const float* first = partials + (size_t)cfirst * cstride +
                             (sc.lo(cfirst) < P0 ? (size_t)rows_per_chunk * PSTRIDE : 0) + (size_t)row * PSTRIDE;
        const float* rest = partials + (size_t)cfirst * cstride + (size_t)row * PSTRIDE;
        auto piece = [&](int i) -> const float* { return i == 0 ? first : rest + (size_t)i * cstride; };
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (np <= MERGE_PIECES) {
            float mv[MERGE_PIECES], lv[MERGE_PIECES];
            float4 ov[MERGE_PIECES];
#pragma unroll
            for (int i = 0; i < MERGE_PIECES; ++i) {
                if (i < np) {
                    const float* pr = piece(i);
                    mv[i] = pr[D];
                    lv[i] = pr[D + 1];
                    ov[i] = *reinterpret_cast<const float4*>(pr + d0);
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < MERGE_PIECES; ++i)
                if (i < np) M = fmaxf(M, mv[i]);
            const float Mref = M == -INFINITY ? 0.f : M;
#pragma unroll
            for (int i = 0; i < MERGE_PIECES; ++i) {
                if (i < np) {
                    const float f = ex2(mv[i] - Mref);
                    L += lv[i] * f;
                    acc.x += ov[i].x * f;
                    acc.y += ov[i].y * f;
                    acc.z += ov[i].z * f;
                    acc.w += ov[i].w * f;
                }
            }
        } else {
            float M = -INFINITY;
            for (int i = 0; i < np; ++i) M = fmaxf(M, piece(i)[D]);
            const float Mref = M == -INFINITY ? 0.f : M;
            for (int i = 0; i < np; ++i) {
                const float* pr = piece(i);
                const float f = ex2(pr[D] - Mref);
                L += pr[D + 1] * f;
                const float4 v = *reinterpret_cast<const float4*>(pr + d0);
                acc.x += v.x * f;
                acc.y += v.y * f;
                acc.z += v.z * f;
                acc.w += v.w * f;
            }
        }
        if (!writer) continue;
        const float inv = 1.f / L;
        const float xv[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
        uint32_t w[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint16_t h0 = bf16 ? f32_to_16<true>(xv[2 * k]) : f32_to_16<false>(xv[2 * k]);
            const uint16_t h1 = bf16 ? f32_to_16<true>(xv[2 * k + 1]) : f32_to_16<false>(xv[2 * k + 1]);
            w[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        }
        uint16_t* dst = out + ((size_t)(qa + rr / G) * Hq + (size_t)kvh * G + rr % G) * D + d0;
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
}

struct MultiLaunch {
    const CUtensorMap* tmap_q;   // tensor-core kernel only: q as [T][Hq][D]
    const CUtensorMap* tmap_k;
    const CUtensorMap* tmap_v;
    MultiParams p;
    cudaStream_t stream;
    int grid;
};

struct MultiKernelInfo {
    cudaError_t (*launch)(const MultiLaunch&);
    int (*max_ctas)(int device);
    int rows;                    // query rows per CTA
};

template <class Tr>
cudaError_t multi_launch(const MultiLaunch& L) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream, attr);
    return cudaLaunchKernelEx(&cfg, pa_multi_kernel<Tr>, *L.tmap_k, *L.tmap_v, L.p);
}

template <class Tr>
MultiKernelInfo multi_info() {
    return MultiKernelInfo{&multi_launch<Tr>, &persistent_ctas<pa_multi_kernel<Tr>, Tr::THREADS, Tr::SMEM_BYTES>,
                           Tr::ROWS};
}

// Index: [bs == 32] (one 16-row tile, NW = 1); one table per (dtype, head_dim), defined in multi_*.cu.
void multi_table_bf16_d128(MultiKernelInfo (&t)[2]);
void multi_table_bf16_d64(MultiKernelInfo (&t)[2]);
void multi_table_fp16_d128(MultiKernelInfo (&t)[2]);
void multi_table_fp16_d64(MultiKernelInfo (&t)[2]);

}  // namespace pa
