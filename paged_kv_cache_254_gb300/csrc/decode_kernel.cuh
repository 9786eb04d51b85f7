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
// contributing ceil(ctx / B) blocks; the flattened block list is cut into
// gridDim.x equal contiguous ranges, one per persistent CTA.  A CTA walks its
// range as "segments" (the part of one pair that falls in the range).  A pair
// that lies inside one CTA is finished there; a pair cut by range boundaries
// leaves a partial softmax state (m, l, unnormalised o) per piece in the
// workspace, and the last CTA to finish a piece of that pair (arrival counter,
// zeroed by the host before the launch) merges them with the log-sum-exp rule
// in CTA order.
// Everything about the split depends on context lengths only, never on block
// ids, so results are bitwise independent of block placement.
//
// Inside a CTA.  Warp NC is the producer: it reads block ids from the table
// (32 at a time, one per lane), and lane 0 issues two-dimensional TMA loads
// (128-byte swizzle) of each (block, KV head) K chunk and V chunk into a ring
// of shared-memory stages guarded by full/empty mbarriers.  Warps 0..NC-1 are
// consumers: within a segment, warp w takes blocks w, w+NC, ...; per block it
// computes S^T = Q K^T for the whole query-head group with mma.sync
// (m16n8k16, fp32 accumulate; heads are the M rows, padded to 16), runs the
// online-softmax update in registers (row max over the lanes of a row by
// shuffles, exp2 with the scale folded into log2(e)), and accumulates
// O^T += V^T P^T with mma.sync, feeding the probabilities straight from the
// score fragments.  At the end of a segment the NC warp states are merged
// through shared memory.
//
// Every wait is bounded (PA_DEVERR_TIMEOUT); bad block ids and context lengths
// set error bits and poison the affected rows with NaN instead of trapping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"
#include "../../include/pa.h"

namespace pa {

struct DecodeParams {
    const uint16_t* q;            // [N][Hq][D]
    const int32_t* block_tables;  // [N][MB]
    const int32_t* context_lens;  // [N]
    uint16_t* out;                // [N][Hq][D]
    int32_t* counters;            // [N * Hkv], zeroed before each launch
    float* partials;              // [gridDim.x][2][G][D + 2]
    uint32_t* err;                // may be null
    int32_t N, Hq, Hkv, NB, MB;
    float scale_log2;             // scale * log2(e)
    uint64_t timeout_ns;
};

template <int D_, int BS_, int G_, bool BF16_>
struct DecodeTraits {
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr int G = G_;
    static constexpr bool BF16 = BF16_;
    static constexpr int NC = 4;                            // consumer warps
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int HALVES = D / 64;                   // 128-byte column boxes per row
    static constexpr int BOX_BYTES = BS * 128;
    static constexpr int CHUNK_BYTES = HALVES * BOX_BYTES;  // one (block, head) chunk
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;     // K + V
    static constexpr int RING_TARGET = 64 * 1024;
    static constexpr int STAGES = (RING_TARGET / STAGE_BYTES) > 16 ? 16 : (RING_TARGET / STAGE_BYTES);
    static constexpr int NR = G > 8 ? 2 : 1;                // 8-row groups of query heads in use
    static constexpr int NT = BS / 8;                       // 8-token n-tiles of S^T
    static constexpr int KT = BS / 16;                      // 16-token k-steps of PV
    static constexpr int KD = D / 16;                       // 16-dim k-steps of QK / m-tiles of PV
    static constexpr int OSTRIDE = D + 4;                   // padded scratch row (bank spread)
    static constexpr int PSTRIDE = D + 2;                   // partial row: o[D], m, l
    // shared memory carve-up, offsets from a 1024-byte aligned base
    static constexpr int RING_OFF = 0;
    static constexpr int SO_OFF = STAGES * STAGE_BYTES;
    static constexpr int SO_BYTES = NC * G * OSTRIDE * 4;
    static constexpr int SM_OFF = SO_OFF + SO_BYTES;        // m per (warp, head)
    static constexpr int SL_OFF = SM_OFF + NC * G * 4;      // l per (warp, head)
    static constexpr int SP_OFF = SL_OFF + NC * G * 4;      // poison flag per warp
    static constexpr int PS_OFF = SP_OFF + NC * 4;          // poison flag per stage
    static constexpr int BAR_OFF = ((PS_OFF + STAGES * 4) + 7) & ~7;
    static constexpr int INFO_OFF = BAR_OFF + 2 * STAGES * 8;
    static constexpr int INFO_BYTES = 64;
    static constexpr int SMEM_BYTES = INFO_OFF + INFO_BYTES + 1024;  // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
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

__device__ __forceinline__ int seq_blocks(int ctx, int BS, int MB) {
    return (ctx > 0 && ctx <= MB * BS) ? (ctx + BS - 1) / BS : 0;
}

// Largest CTA index c with floor(c * W / G) <= x.
__device__ __forceinline__ long long cta_of(long long x, long long W, long long G) {
    return ((x + 1) * G + W - 1) / W - 1;
}

__device__ __forceinline__ long long range_lo(long long c, long long W, long long G) {
    return c * W / G;
}

// Position inside the flattened block list, advanced segment by segment.
struct SegIter {
    long long gi;  // flattened index of the next block
    int s, kvh, b0, nb;
};

__device__ __forceinline__ void seg_advance(SegIter& it, int len, const DecodeParams& p, int BS) {
    it.gi += len;
    it.b0 += len;
    if (it.b0 == it.nb) {
        it.b0 = 0;
        if (++it.kvh == p.Hkv) {
            it.kvh = 0;
            int nb = 0;
            while (++it.s < p.N) {
                nb = seq_blocks(__ldg(p.context_lens + it.s), BS, p.MB);
                if (nb > 0) break;
            }
            it.nb = nb;
        }
    }
}

template <class Tr>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)((chunk >> 3) * Tr::BOX_BYTES + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

template <bool BF16>
__device__ __forceinline__ uint16_t f32_to_16(float x) {
    if constexpr (BF16) {
        uint16_t r;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
        return r;
    } else {
        uint16_t r;
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
        return r;
    }
}

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, 2)
pa_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const DecodeParams p) {
    constexpr int D = Tr::D, BS = Tr::BS, G = Tr::G, NC = Tr::NC, S = Tr::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(smem + Tr::RING_OFF);
    float* so = reinterpret_cast<float*>(smem + Tr::SO_OFF);
    float* sm = reinterpret_cast<float*>(smem + Tr::SM_OFF);
    float* sl = reinterpret_cast<float*>(smem + Tr::SL_OFF);
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
    if (warp == NC && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }

    // ---- work range of this CTA (warp 0) ----
    if (warp == 0) {
        long long w = 0;
        for (int s = lane; s < p.N; s += 32) w += seq_blocks(__ldg(p.context_lens + s), BS, p.MB);
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
                const long long v = s < p.N ? (long long)seq_blocks(__ldg(p.context_lens + s), BS, p.MB) * p.Hkv : 0;
                long long incl = v;
                for (int o = 1; o < 32; o <<= 1) {
                    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const long long total = __shfl_sync(0xffffffffu, incl, 31);
                if (base + total > lo) {
                    const unsigned m = __ballot_sync(0xffffffffu, base + incl > lo);
                    const int first = __ffs(m) - 1;
                    const long long before = base + __shfl_sync(0xffffffffu, incl - v, first);
                    s0 = sb + first;
                    const int nb = seq_blocks(__ldg(p.context_lens + s0), BS, p.MB);
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

    // ---- rows of sequences with no blocks: zero (ctx == 0) or NaN (bad ctx) ----
    if (warp < NC) {
        for (int s = blockIdx.x; s < p.N; s += gridDim.x) {
            const int ctx = __ldg(p.context_lens + s);
            if (ctx > 0 && ctx <= p.MB * BS) continue;
            const bool bad = ctx != 0;
            if (bad && threadIdx.x == 0) set_err(p.err, PA_DEVERR_CONTEXT);
            const uint16_t v = bad ? (Tr::BF16 ? (uint16_t)0x7fc0 : (uint16_t)0x7e00) : (uint16_t)0;
            uint16_t* row = p.out + (size_t)s * p.Hq * D;
            for (int i = threadIdx.x; i < p.Hq * D; i += NC * 32) row[i] = v;
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
    it0.nb = seq_blocks(__ldg(p.context_lens + it0.s), BS, p.MB);

    if (warp == NC) {
        // =========================== producer ===========================
        long long issued = 0;
        bool aborted = false;
        SegIter it = it0;
        while (it.gi < hi && !aborted) {
            const int len = (int)min((long long)(it.nb - it.b0), hi - it.gi);
            const int32_t* trow = p.block_tables + (size_t)it.s * p.MB + it.b0;
            int tcur = lane < len ? __ldg(trow + lane) : 0;
            for (int base = 0; base < len && !aborted; base += 32) {
                const int nxt = base + 32 + lane < len ? __ldg(trow + base + 32 + lane) : 0;
                const int cnt = min(32, len - base);
                for (int i = 0; i < cnt; ++i) {
                    int id = __shfl_sync(0xffffffffu, tcur, i);
                    int ok = 1;
                    if (lane == 0) {
                        const int st = (int)(issued % S);
                        if (issued >= S) {
                            const uint32_t par = (uint32_t)(((issued / S) - 1) & 1);
                            if (!mbar_wait_bounded(empty0 + 8 * st, par, p.timeout_ns)) ok = 0;
                        }
                        if (ok) {
                            const bool bad = (unsigned)id >= (unsigned)p.NB;
                            if (bad) {
                                set_err(p.err, PA_DEVERR_BLOCK_ID);
                                id = 0;
                            }
                            stage_poison[st] = bad ? 1 : 0;
                            const uint32_t fb = full0 + 8 * st;
                            mbar_arrive_expect_tx(fb, Tr::STAGE_BYTES);
                            const int y = (id * p.Hkv + it.kvh) * BS;
                            const uint32_t kdst = ring_u32 + st * Tr::STAGE_BYTES;
#pragma unroll
                            for (int h = 0; h < Tr::HALVES; ++h) {
                                tma_load_2d(kdst + h * Tr::BOX_BYTES, &tmap_k, h * 64, y, fb);
                                tma_load_2d(kdst + Tr::CHUNK_BYTES + h * Tr::BOX_BYTES, &tmap_v, h * 64, y, fb);
                            }
                        } else {
                            set_err(p.err, PA_DEVERR_TIMEOUT);
                            *(volatile int*)&info->abort = 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        aborted = true;
                        break;
                    }
                    ++issued;
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
    while (it.gi < hi) {
        const int len = (int)min((long long)(it.nb - it.b0), hi - it.gi);
        const int ctx = __ldg(p.context_lens + it.s);

        // Q fragments (A operand of S^T = Q K^T): rows = heads of the group.
        const uint16_t* qrow = p.q + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * D;
        uint32_t qa[Tr::KD][4];
#pragma unroll
        for (int kk = 0; kk < Tr::KD; ++kk) {
            const int c = kk * 16 + 2 * t4;
            qa[kk][0] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(qrow + g * D + c)) : 0u;
            qa[kk][2] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(qrow + g * D + c + 8)) : 0u;
            if constexpr (G > 8) {
                qa[kk][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + (g + 8) * D + c));
                qa[kk][3] = __ldg(reinterpret_cast<const uint32_t*>(qrow + (g + 8) * D + c + 8));
            } else {
                qa[kk][1] = 0u;
                qa[kk][3] = 0u;
            }
        }

        float m_run[Tr::NR], l_run[Tr::NR];
        float o[Tr::KD][Tr::NR][4];
#pragma unroll
        for (int r = 0; r < Tr::NR; ++r) {
            m_run[r] = -INFINITY;
            l_run[r] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < Tr::KD; ++mt)
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][r][e] = 0.f;
        int poisoned = 0;

        // Block k of the CTA range (k = gi - lo) goes to warp k % NC.  With
        // STAGES a multiple of NC every ring stage is owned by one warp, which
        // consumes its fills strictly in order (no mbarrier phase aliasing).
        int j0 = warp - (int)((it.gi - lo) % NC);
        if (j0 < 0) j0 += NC;
        for (int j = j0; j < len; j += NC) {
            const long long k = it.gi + j - lo;
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
            const int valid = min(BS, ctx - (it.b0 + j) * BS);
            const uint32_t kb = ring_u32 + st * Tr::STAGE_BYTES;
            const uint32_t vb = kb + Tr::CHUNK_BYTES;

            // ---- S^T = Q K^T : [16 heads x BS tokens] ----
            float sacc[Tr::NT][4];
#pragma unroll
            for (int nt = 0; nt < Tr::NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < Tr::KD / 2; ++q4) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + swz<Tr>(nt * 8 + (lane & 7), q4 * 4 + (lane >> 3)), b0, b1, b2, b3);
                    mma16816<Tr::BF16>(sacc[nt], qa[2 * q4][0], qa[2 * q4][1], qa[2 * q4][2], qa[2 * q4][3], b0, b1);
                    mma16816<Tr::BF16>(sacc[nt], qa[2 * q4 + 1][0], qa[2 * q4 + 1][1], qa[2 * q4 + 1][2],
                                       qa[2 * q4 + 1][3], b2, b3);
                }
            }

            // ---- scale, mask tokens past the context, online softmax ----
            float mx[Tr::NR];
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r) mx[r] = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < Tr::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = nt * 8 + 2 * t4 + (e & 1);
                    const float v = tok < valid ? sacc[nt][e] * p.scale_log2 : -INFINITY;
                    sacc[nt][e] = v;
                    if ((e >> 1) < Tr::NR) mx[e >> 1] = fmaxf(mx[e >> 1], v);
                }
            float alpha[Tr::NR];
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float m_new = fmaxf(m_run[r], mx[r]);
                alpha[r] = ex2(m_run[r] - m_new);
                m_run[r] = m_new;
                l_run[r] *= alpha[r];
            }
#pragma unroll
            for (int nt = 0; nt < Tr::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1;
                    if (r < Tr::NR) {
                        const float pe = ex2(sacc[nt][e] - m_run[r]);
                        sacc[nt][e] = pe;
                        l_run[r] += pe;
                    }
                }
            // P^T fragments (B operand of O^T += V^T P^T): k = tokens, n = heads.
            // P is carried as hi + lo, two 16-bit parts (hi = round(p),
            // lo = round(p - hi)), so the product keeps ~16 bits of p instead
            // of the 8 a single bf16 would leave.
            uint32_t pb[Tr::KT][Tr::NR][2], pl[Tr::KT][Tr::NR][2];
#pragma unroll
            for (int kt = 0; kt < Tr::KT; ++kt)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float x0 = sacc[2 * kt + h][2 * r], x1 = sacc[2 * kt + h][2 * r + 1];
                        const uint32_t hi = pack2<Tr::BF16>(x0, x1);
                        pb[kt][r][h] = hi;
                        pl[kt][r][h] = pack2<Tr::BF16>(x0 - lo_of<Tr::BF16>(hi), x1 - hi_of<Tr::BF16>(hi));
                    }

            // Rows past the context in a partly filled block may hold anything
            // (even NaN); zero them so 0 * V stays 0 in the PV product.
            if (valid < BS) {
                const int nz = (BS - valid) * Tr::HALVES * 8;   // 16-byte pieces
                for (int i = lane; i < nz; i += 32) {
                    const int piece = i & 7;
                    const int rest = i >> 3;
                    const int h = rest % Tr::HALVES;
                    const int row = valid + rest / Tr::HALVES;
                    const uint32_t a = vb + h * Tr::BOX_BYTES + row * 128 + piece * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(a), "r"(0) : "memory");
                }
                __syncwarp();
            }

            // ---- rescale the running O^T by exp2(m_old - m_new) per head ----
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r) {
                const float aa = __shfl_sync(0xffffffffu, alpha[r], (2 * t4) * 4);
                const float ab = __shfl_sync(0xffffffffu, alpha[r], (2 * t4 + 1) * 4);
#pragma unroll
                for (int mt = 0; mt < Tr::KD; ++mt) {
                    o[mt][r][0] *= aa;
                    o[mt][r][1] *= ab;
                    o[mt][r][2] *= aa;
                    o[mt][r][3] *= ab;
                }
            }

            // ---- O^T[d x heads] += V^T[d x tokens] P^T[tokens x heads] ----
#pragma unroll
            for (int mt = 0; mt < Tr::KD; ++mt)
#pragma unroll
                for (int kt = 0; kt < Tr::KT; ++kt) {
                    uint32_t a0, a1, a2, a3;
                    const int row = kt * 16 + ((lane >> 4) << 3) + (lane & 7);
                    const int chunk = 2 * mt + ((lane >> 3) & 1);
                    ldsm_x4_t(vb + swz<Tr>(row, chunk), a0, a1, a2, a3);
#pragma unroll
                    for (int r = 0; r < Tr::NR; ++r) {
                        mma16816<Tr::BF16>(o[mt][r], a0, a1, a2, a3, pb[kt][r][0], pb[kt][r][1]);
                        mma16816<Tr::BF16>(o[mt][r], a0, a1, a2, a3, pl[kt][r][0], pl[kt][r][1]);
                    }
                }
            if (valid < BS) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }

        // ---- merge the NC warp states of this segment ----
#pragma unroll
        for (int r = 0; r < Tr::NR; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
        {
            float* mine = so + warp * G * Tr::OSTRIDE;
#pragma unroll
            for (int mt = 0; mt < Tr::KD; ++mt)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int head = 8 * r + 2 * t4 + (e & 1);
                        const int dim = 16 * mt + g + 8 * (e >> 1);
                        if (head < G) mine[head * Tr::OSTRIDE + dim] = o[mt][r][e];
                    }
            if (t4 == 0) {
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r) {
                    const int head = g + 8 * r;
                    if (head < G) {
                        sm[warp * G + head] = m_run[r];
                        sl[warp * G + head] = l_run[r];
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
        int bad = 0;
#pragma unroll
        for (int w = 0; w < NC; ++w) bad |= spois[w];
        const float qnan = __int_as_float(0x7fc00000);
        uint16_t* orow = p.out + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * D;
        float* prow = p.partials + ((size_t)blockIdx.x * 2 + slot) * G * Tr::PSTRIDE;
        for (int idx = tid; idx < G * D; idx += NC * 32) {
            const int head = idx / D;
            const int dim = idx - head * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NC; ++w) M = fmaxf(M, sm[w * G + head]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                const float f = ex2(sm[w * G + head] - M);
                L += sl[w * G + head] * f;
                O += so[(w * G + head) * Tr::OSTRIDE + dim] * f;
            }
            if (bad) O = qnan;
            if (complete) {
                orow[head * D + dim] = f32_to_16<Tr::BF16>(O / L);
            } else {
                prow[head * Tr::PSTRIDE + dim] = O;
                if (dim == 0) {
                    prow[head * Tr::PSTRIDE + D] = M;
                    prow[head * Tr::PSTRIDE + D + 1] = L;
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
                        const float mc = __ldcg(pr + D);
                        const float lc = __ldcg(pr + D + 1);
                        const float oc = __ldcg(pr + dim);
                        const float Mn = fmaxf(M, mc);
                        const float fa = ex2(M - Mn), fb = ex2(mc - Mn);
                        L = L * fa + lc * fb;
                        O = O * fa + oc * fb;
                        M = Mn;
                    }
                    orow[head * D + dim] = f32_to_16<Tr::BF16>(O / L);
                }
            }
        }
        named_bar_sync(1, NC * 32);
        seg_advance(it, len, p, BS);
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
int decode_max_ctas(int device) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return -1;
    if (cached[device] > 0) return cached[device];
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return -1;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return -1;
    int sms = 0, per_sm = 0;
    cudaError_t e = cudaFuncSetAttribute(pa_decode_kernel<Tr>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tr::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_decode_kernel<Tr>, Tr::THREADS,
                                                          Tr::SMEM_BYTES);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || per_sm <= 0) return -1;
    cached[device] = sms * per_sm;
    return cached[device];
}

template <class Tr>
DecodeKernelInfo decode_info() {
    return DecodeKernelInfo{&decode_launch<Tr>, &decode_max_ctas<Tr>, Tr::SMEM_BYTES, Tr::STAGES};
}

// Per-(dtype, head_dim) tables, defined in the instantiation units.
// Index: [bs == 32][log2(g)].
void decode_table_bf16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_bf16_d64(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d64(DecodeKernelInfo (&t)[2][5]);

}  // namespace pa
