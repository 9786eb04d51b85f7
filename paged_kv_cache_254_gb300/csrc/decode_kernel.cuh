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
// contributing its blocks; the flattened block list is cut into contiguous
// chunks.  A worker is one warp of a persistent CTA, and works alone: it
// walks its chunks as "segments" (the part of one pair that falls in a
// chunk), keeping the online-softmax state of the pair's query rows in its
// registers.  The first three quarters of the list form one chunk per worker
// (worker w takes chunk w); the last quarter is cut into `nd` small chunks
// that workers claim with an atomic counter when they run out, which evens
// out SMs that get less memory bandwidth or more segment ends than others.
// A pair that lies inside one chunk is finished by its warp; a pair cut by
// chunk boundaries leaves a partial state (m, l, unnormalised o) per piece in
// the workspace, and a post-pass kernel (pa_decode_merge, one warp per pair
// and query head, launched to wait on this grid with griddepcontrol) merges
// the pieces with the log-sum-exp rule in chunk order, so no warp ever waits
// on another.  Chunk boundaries depend on context lengths and the grid only, never
// on block ids or on which warp took a chunk, so results are bitwise
// independent of block placement and of timing.  A chunk start is found by a
// search over per-sequence block prefix sums (written by a pre-pass kernel,
// copied to shared memory when there are at most CUM_SMEM sequences).
//
// Shared prefixes (optional).  With prefix groups, the first first_blocks[s]
// blocks of a member sequence were already reduced by the prefix kernel into
// a per-row state (the carry); here the pair covers only the sequence's own
// blocks after the prefix, and the carry joins the final log-sum-exp
// combination.
//
// Inside a warp.  Each warp owns R shared-memory stages with one mbarrier
// each.  The copies of a stage (one 3-D TMA box with 128-byte swizzle per
// block for K and one for V in the 16-bit cache, one bulk copy per block
// piece for the quantized caches, all under an L2 evict-first policy: the
// stream is read once) are issued R stages ahead of the one being computed, and
// a stage is refilled as soon as it has been folded in (mma.sync scores,
// online softmax, PV: consume_block for the 16-bit cache with the query heads
// as MMA rows; consume_stage8t / consume_stage4t for the quantized caches
// with the stage's tokens as MMA rows).  Block ids come from the table 32 at
// a time, one per lane.  No warp ever waits for another.
//
// Every wait is bounded (PA_DEVERR_TIMEOUT); bad block ids and context lengths
// set error bits and poison the affected rows with NaN instead of trapping.
#pragma once

#include <type_traits>

#include "decode_common.cuh"
#include "decode_tok.cuh"

namespace pa {

struct DecodeParams {
    const uint16_t* q;            // [N][Hq][D]
    const int32_t* block_tables;  // [N][MB]
    const int32_t* context_lens;  // [N]
    uint16_t* out;                // [N][Hq][D]
    float* partials;              // [chunks][2][G][D + 4]
    uint32_t* err;                // may be null
    // shared prefixes (first_blocks == null: none)
    const int32_t* first_blocks;  // [N] blocks already covered by the prefix pass
    const float* carry;           // [N][Hq][D + 2] prefix states (o, m, l)
    const uint8_t* kv8;           // 8-bit cache only: the pool (K rows, then dims-first V, per piece)
    float v_scale;                // multiplies the output (V's cache scale; 1 for 16-bit)
    const long long* cum;         // [N + 1] blocks of sequences before s (pre-pass)
    int32_t* chunk_ctr;           // dynamic chunks claimed so far (zeroed by the pre-pass)
    int32_t nd;                   // dynamic chunks wanted (0: the static split alone)
    int32_t N, Hq, Hkv, NB, MB;
    float scale_log2;             // scale * log2(e)
    uint64_t timeout_ns;          // limit of every wait on copies
    // Fault injection for tests (0: off): each worker's first stage wait is
    // made on a barrier that nothing completes, bounded by stall_ns, so the
    // timeout path runs; the drain of copies in flight keeps timeout_ns.
    uint64_t stall_ns;
};

// Bytes of pool data a full stage holds (without bank padding).
template <class Gm, bool KV8>
constexpr int stage_data_bytes() {
    if constexpr (KV8) {
        return Gm::COPY_BYTES;
    } else {
        return Gm::STAGE_BYTES;
    }
}

// KVF: 0 = the cache holds q's 16-bit type; 1 = FP8 E4M3 codes; 2 = FP8 E5M2;
// 3 = 4-bit integer codes with per-row scales.  KV8: any quantized cache (one
// contiguous piece per (block, head), fetched by bulk copies).
template <int D_, int BS_, int G_, bool BF16_, int KVF_ = 0>
struct DecodeTraits {
    static constexpr bool KV8 = KVF_ != 0;
    static constexpr bool I4 = KVF_ == 3;
    using Gm = std::conditional_t<I4, Geom4<BS_>, std::conditional_t<KV8, Geom8<BS_>, Geom<D_, BS_>>>;
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr int UB = Gm::UB;                       // blocks per stage
    static constexpr int G = G_;
    static constexpr bool BF16 = BF16_;
    static constexpr bool E5M2 = KVF_ == 2;
    // About 192 KiB of stages per SM (200 KiB for the quantized caches, whose
    // two-piece stages carry 64 bytes of bank padding): stages of up to 8 KiB
    // of data, two CTAs of four warps; 16 KiB stages, one CTA of six warps.
    // The 4-bit cache: 64-token stages (8.6 KiB), two CTAs of four warps with
    // three stages each (212 KB of copies in flight per SM).
    static constexpr int RING_PER_SM = (KV8 ? 200 : 192) * 1024;
    static constexpr int DATA_BYTES = stage_data_bytes<Gm, KV8>();
    static constexpr int MIN_CTAS = I4 ? 2 : DATA_BYTES <= 8192 ? 2 : 1;
    static constexpr int NW = MIN_CTAS == 1 ? 6 : 4;       // warps (workers) per CTA
    static constexpr int R_FIT = RING_PER_SM / (MIN_CTAS * NW * Gm::STAGE_BYTES);
    // stages per warp (the 4-bit cache: see above)
    static constexpr int R = I4 ? 3 : R_FIT > 8 ? 8 : R_FIT;
    static constexpr int THREADS = NW * 32;
    static constexpr int NR = G > 8 ? 2 : 1;                // 8-row groups of query heads in use
    // quantized caches: the stage's tokens are the MMA rows (decode_tok.cuh)
    static constexpr bool TR = KV8;
    using Acc = std::conditional_t<TR, WarpAccT<D_, NR>, WarpAcc<D_, NR>>;
    static constexpr int PSTRIDE = D_ + 4;                  // partial row: o[D], m, l, 2 pad (16-byte rows)
    static constexpr int CSTRIDE = D_ + 2;                  // carry row (prefix pass): o[D], m, l
    static constexpr int CUM_SMEM = I4 ? 256 : 512;         // sequences whose tables fit in smem
    static constexpr int QN = R + 2 <= 8 ? 8 : 16;          // open chunks per warp (> R + 1)
    // smem base alignment: 1024 for the 128-byte swizzled tensor copies of the
    // 16-bit cache, 128 for the plain bulk copies of the quantized ones
    static constexpr int ALIGN = KV8 ? 128 : 1024;
    // shared memory, offsets from a 1024-byte aligned base
    static constexpr int BAR_OFF = NW * R * Gm::STAGE_BYTES;
    static constexpr int CUM_OFF = BAR_OFF + NW * R * 8;    // long long [CUM_SMEM + 1]
    static constexpr int CTX_OFF = CUM_OFF + (CUM_SMEM + 1) * 8;   // int [CUM_SMEM] context lengths
    static constexpr int FST_OFF = CTX_OFF + CUM_SMEM * 4;  // int [CUM_SMEM] first blocks
    static constexpr int CQ_OFF = FST_OFF + CUM_SMEM * 4;
    static constexpr int PS_OFF = CQ_OFF + NW * QN * 32;    // poison flag per stage
    static constexpr int STALL_OFF = (PS_OFF + NW * R * 4 + 7) & ~7;   // barrier nothing completes (tests)
    static constexpr int SMEM_BYTES = STALL_OFF + 8 + ALIGN;  // + alignment slack
    static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "group size");
    static_assert(R >= 2, "two stages per warp at least");
    static_assert(32 % UB == 0, "a batch of 32 table entries holds whole stages");
};

// Per-sequence data of the work list (in shared memory for small batches):
// cum[s] = blocks of the sequences before s, context lengths, first blocks
// (blocks already covered by a shared-prefix pass; null: none).
struct SeqTab {
    const long long* cum;
    const int* ctx;
    const int* first;
    __device__ __forceinline__ int nb(int s) const { return (int)(cum[s + 1] - cum[s]); }
    __device__ __forceinline__ int fst(int s) const { return first ? first[s] : 0; }
};

// Position inside the flattened block list, advanced segment by segment.
struct SegIter {
    long long gi;  // flattened index of the next block
    int s, kvh, b0, nb, first;
};

__device__ __forceinline__ void seg_advance(SegIter& it, int len, const DecodeParams& p, const SeqTab& tab) {
    it.gi += len;
    it.b0 += len;
    if (it.b0 == it.nb) {
        it.b0 = 0;
        if (++it.kvh == p.Hkv) {
            it.kvh = 0;
            int nb = 0;
            while (++it.s < p.N) {
                nb = tab.nb(it.s);
                if (nb > 0) break;
            }
            it.nb = nb;
            it.first = it.s < p.N ? tab.fst(it.s) : 0;
        }
    }
}

__device__ __forceinline__ int seg_len(const SegIter& it, long long hi) {
    return (int)min((long long)(it.nb - it.b0), hi - it.gi);
}

// Chunks of the flattened list: NS static ones over [0, Ws), then ND over [Ws, W).
struct Sched {
    long long W, Ws;
    int NS, ND;
    __device__ long long lo(long long c) const {
        if (c <= NS) return range_lo(c, Ws, NS);
        return Ws + range_lo(c - NS, W - Ws, ND);
    }
    __device__ long long of(long long x) const {   // the chunk holding flattened block x
        if (x < Ws) return cta_of(x, Ws, NS);
        return NS + cta_of(x - Ws, W - Ws, ND);
    }
};

// The schedule of W flattened blocks over `nworkers` warps with `nd` dynamic
// chunks wanted: the last quarter goes dynamic when every chunk can hold a
// few blocks, else the static split alone.
__device__ __forceinline__ Sched make_sched(long long W, long long nworkers, int nd) {
    Sched sc;
    sc.W = W;
    if (nd > 0 && W >= 64 * nworkers) {
        sc.Ws = W - W / 4;
        sc.NS = (int)nworkers;
        sc.ND = nd;
    } else {
        sc.Ws = W;
        sc.NS = (int)(W < nworkers ? W : nworkers);
        sc.ND = 0;
    }
    return sc;
}

// An open chunk, queued by the issue side for the compute side of one warp.
struct ChunkEnt {
    long long lo, hi;
    int id, s, kvh, b0;
};
static_assert(sizeof(ChunkEnt) <= 32, "chunk queue entry");

// Position of flattened block x (0 <= x < W): the pair (s, kvh) and block b0.
// cum[s] counts the blocks of sequences before s; a 32-way search, one probe
// per lane per round.
__device__ __forceinline__ SegIter locate(const DecodeParams& p, const SeqTab& tab, long long x, int lane) {
    const long long* cum = tab.cum;
    int a = 0, b = p.N;   // cum[a] * Hkv <= x < cum[b] * Hkv
    while (b - a > 1) {
        const int step = (b - a + 31) / 32;
        const int idx = a + lane * step;
        const bool le = idx < b && cum[idx] * p.Hkv <= x;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        const int top = 31 - __clz(m);                 // lane 0 always probes a
        a = a + top * step;
        b = min(a + step, b);
    }
    SegIter it;
    const long long c0 = cum[a];
    const int nb = (int)(cum[a + 1] - c0);
    const long long off = x - c0 * p.Hkv;
    it.gi = x;
    it.s = a;
    it.kvh = (int)(off / nb);
    it.b0 = (int)(off % nb);
    it.nb = nb;
    it.first = tab.fst(a);
    return it;
}

template <class Tr>
__global__ void __launch_bounds__(Tr::THREADS, Tr::MIN_CTAS)
pa_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const DecodeParams p) {
    using Gm = typename Tr::Gm;
    constexpr int D = Tr::D, BS = Tr::BS, G = Tr::G, NW = Tr::NW, R = Tr::R, UB = Tr::UB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + (Tr::ALIGN - 1)) &
                                               ~uintptr_t(Tr::ALIGN - 1));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;       // fragment row group
    const int t4 = lane & 3;       // fragment column pair
    const uint32_t ring = smem_u32(smem) + warp * R * Gm::STAGE_BYTES;      // this warp's stages
    const uint32_t full0 = smem_u32(smem + Tr::BAR_OFF) + warp * R * 8;
    volatile int* stage_poison = reinterpret_cast<volatile int*>(smem + Tr::PS_OFF) + warp * R;

    long long* scum = reinterpret_cast<long long*>(smem + Tr::CUM_OFF);
    int* sctx = reinterpret_cast<int*>(smem + Tr::CTX_OFF);
    int* sfst = reinterpret_cast<int*>(smem + Tr::FST_OFF);
    ChunkEnt* cq = reinterpret_cast<ChunkEnt*>(smem + Tr::CQ_OFF) + warp * Tr::QN;

    const uint32_t stall_bar = smem_u32(smem + Tr::STALL_OFF);
    if (lane == 0) {
        for (int st = 0; st < R; ++st) mbar_init(full0 + 8 * st, 1);
        if (warp == 0) mbar_init(stall_bar, 1);
        fence_mbar_init();
        if constexpr (!Tr::KV8) {
            if (warp == 0) {
                prefetch_tmap(&tmap_k);
                prefetch_tmap(&tmap_v);
            }
        }
    }
    // Everything above is CTA-local; the pre-pass's outputs (and whatever the
    // stream wrote before it) are read only after the previous kernel is done.
    griddep_wait();
    // The merge post-pass may be scheduled now: its CTAs take SMs as this
    // grid's CTAs retire and wait (griddepcontrol.wait) for the whole grid.
    griddep_launch_dependents();
    const bool in_smem = p.N <= Tr::CUM_SMEM;
    if (in_smem) {
        for (int i = threadIdx.x; i <= p.N; i += Tr::THREADS) {
            scum[i] = __ldg(p.cum + i);
            if (i < p.N) {
                sctx[i] = __ldg(p.context_lens + i);
                if (p.first_blocks) sfst[i] = __ldg(p.first_blocks + i);
            }
        }
    }
    __syncthreads();
    SeqTab tab;
    tab.cum = in_smem ? scum : p.cum;
    tab.ctx = in_smem ? sctx : p.context_lens;
    tab.first = p.first_blocks ? (in_smem ? sfst : p.first_blocks) : nullptr;
    const long long* cum = tab.cum;

    // ---- rows of sequences with no blocks here: zero (ctx == 0), the prefix
    //      state alone (every key in a shared prefix), NaN (bad ctx) ----
    for (int s = blockIdx.x; s < p.N; s += gridDim.x) {
        if (cum[s + 1] > cum[s]) continue;
        const int ctx = tab.ctx[s];
        const int first = tab.fst(s);
        const bool bad = ctx < 0 || ctx > p.MB * BS;
        if (bad && threadIdx.x == 0) set_err(p.err, PA_DEVERR_CONTEXT);
        uint16_t* row = p.out + (size_t)s * p.Hq * D;
        for (int i = threadIdx.x; i < p.Hq * D; i += Tr::THREADS) {
            uint16_t v = 0;
            if (bad) {
                v = qnan16<Tr::BF16>();
            } else if (first > 0 && ctx > 0) {
                const float* c = p.carry + ((size_t)s * p.Hq + i / D) * Tr::CSTRIDE;
                v = f32_to_16<Tr::BF16>(__ldg(c + i % D) / __ldg(c + D + 1) * p.v_scale);
            }
            row[i] = v;
        }
    }

    // ---- the chunk schedule ----
    const long long nworkers = (long long)gridDim.x * NW;
    const long long wid = (long long)blockIdx.x * NW + warp;
    const Sched sc = make_sched(cum[p.N] * p.Hkv, nworkers, p.nd);
    const int nchunks = sc.NS + sc.ND;
    if (nchunks == 0) return;
    // next chunk for this warp: its static one first, then claims (lane 0's
    // claim is made one chunk ahead so its latency stays hidden)
    int claim = 0;
    auto claim_async = [&]() {
        if (sc.ND > 0 && lane == 0) claim = sc.NS + atomicAdd(p.chunk_ctr, 1);
        else claim = nchunks;
    };
    int next_id;
    if (wid < sc.NS) {
        next_id = (int)wid;
    } else {
        claim_async();
        next_id = __shfl_sync(0xffffffffu, claim, 0);
    }
    if (next_id >= nchunks) return;
    claim_async();
    int qhead = 0, qtail = 0;   // chunk queue: pushed by the issue side, popped by the compute side

    // ---- issue side: runs up to R stages ahead of the compute side ----
    // Block ids come from the table 32 at a time (one per lane): tcur holds
    // entries [row_off, row_off + 32) of sequence row_s's row, tnxt the next
    // 32.  The KV heads of a sequence share its row, so a batch is reused
    // across them; the first batch of the next sequence is fetched (tpre)
    // while the current one is in use.
    SegIter is{};             // set by open_chunk before the first issue
    // the KV stream is read once: its L2 lines go first, so the partial
    // states written meanwhile are still in L2 when the merge reads them
    const uint64_t kv_pol = l2_evict_first();
    long long ihi = 0;
    int ilen = 0, ib = 0, tbase = 0;
    int tcur = 0, tnxt = 0, tpre = 0;
    int row_s = -1, row_off = 0, pre_s = -1;
    bool idone = false;
    auto row_ids = [&](int sq, int off, int navail) -> int {
        return lane < navail ? __ldg(p.block_tables + (size_t)sq * p.MB + off + lane) : 0;
    };
    // the table batch for the segment starting at `is`
    auto seg_ids = [&]() {
        const int off = is.first + is.b0;
        ib = 0;
        tbase = 0;
        if (!(is.s == row_s && off == row_off)) {
            if (is.s == pre_s && is.b0 == 0) {
                tcur = tpre;
            } else {
                tcur = row_ids(is.s, off, is.nb - is.b0);
            }
            tnxt = row_ids(is.s, off + 32, is.nb - is.b0 - 32);
            row_s = is.s;
            row_off = off;
            // the next sequence with blocks, from its first entry
            int sn = is.s + 1;
            while (sn < p.N && tab.nb(sn) == 0) ++sn;
            pre_s = sn < p.N ? sn : -1;
            if (pre_s >= 0) tpre = row_ids(sn, tab.fst(sn), tab.nb(sn));
        }
        ilen = seg_len(is, ihi);
    };
    // open chunk `id`: locate its start, queue it for the compute side
    auto open_chunk = [&](int id) {
        const long long clo = sc.lo(id);
        ihi = sc.lo(id + 1);
        is = locate(p, tab, clo, lane);
        if (lane == 0) {
            ChunkEnt& e = cq[qtail % Tr::QN];
            e.lo = clo;
            e.hi = ihi;
            e.id = id;
            e.s = is.s;
            e.kvh = is.kvh;
            e.b0 = is.b0;
        }
        ++qtail;
        seg_ids();
    };
    open_chunk(next_id);
    long long nis = 0;        // stages issued
    long long nreal = 0;      // of which with copies (all of them until an abort)
    int ist = 0;              // ring stage of the next fill (nis % R, kept without a division)
    bool aborted = false;     // warp-uniform
    // After an abort the walk goes on without copies, so every chunk is still
    // opened, and every row and partial state of this worker is written (NaN).
    auto issue = [&]() {
        if (idone) return;
        const int st = ist;
        if (++ist == R) ist = 0;
        const int nblk = min(UB, ilen - ib);
        int ids[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) ids[u] = __shfl_sync(0xffffffffu, tcur, (ib - tbase + u) & 31);
        if (lane == 0 && !aborted) {
            bool bad = false;
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                if (u < nblk && (unsigned)ids[u] >= (unsigned)p.NB) {
                    bad = true;
                    ids[u] = 0;
                }
            }
            if (bad) set_err(p.err, PA_DEVERR_BLOCK_ID);
            stage_poison[st] = bad ? 1 : 0;
            if constexpr (Tr::KV8) {
                mbar_arrive_expect_tx(full0 + 8 * st, nblk * Gm::PIECE_BYTES);
            } else {
                mbar_arrive_expect_tx(full0 + 8 * st, Gm::STAGE_BYTES);
            }
        }
        if constexpr (Tr::KV8) {
            // each block's piece is one contiguous run in the pool: one bulk
            // copy per piece, lane u issuing piece u (each copy instruction
            // holds its issuing thread a while; lanes issue side by side)
            __syncwarp();
            if (!aborted && lane < nblk) {
                int id = 0;
#pragma unroll
                for (int u = 0; u < UB; ++u)
                    if (u == lane) id = ids[u];
                if ((unsigned)id >= (unsigned)p.NB) id = 0;   // flagged by lane 0 above
                bulk_load_hint(ring + st * Gm::STAGE_BYTES + Gm::poff(lane),
                               p.kv8 + ((size_t)id * p.Hkv + is.kvh) * Gm::PIECE_BYTES, Gm::PIECE_BYTES,
                               full0 + 8 * st, kv_pol);
            }
        } else {
            // the block's K and V chunks, one 3-D box each ([column half][BS
            // rows][128 B]), issued by two lanes side by side (the TMA unit's
            // cost is per box, and each instruction holds its thread a while)
            __syncwarp();
            if (!aborted && lane < 2) {
                const int id = (unsigned)ids[0] < (unsigned)p.NB ? ids[0] : 0;   // a bad id is flagged above
                tma_load_3d_hint(ring + st * Gm::STAGE_BYTES + (lane ? Gm::CHUNK_BYTES : 0),
                                 lane ? &tmap_v : &tmap_k, 0, (id * p.Hkv + is.kvh) * BS, 0, full0 + 8 * st, kv_pol);
            }
        }
        ++nis;
        if (!aborted) nreal = nis;
        ib += nblk;
        if (ib == ilen) {
            seg_advance(is, ilen, p, tab);
            if (is.gi < ihi) {
                seg_ids();
            } else {
                const int nid = __shfl_sync(0xffffffffu, claim, 0);
                if (nid < nchunks) {
                    claim_async();
                    open_chunk(nid);
                } else {
                    idone = true;
                }
            }
        } else if (ib - tbase == 32) {
            tbase += 32;
            row_off += 32;
            tcur = tnxt;
            tnxt = row_ids(is.s, is.first + is.b0 + tbase + 32, is.nb - is.b0 - tbase - 32);
        }
    };
    for (int i = 0; i < R; ++i) issue();

    // ---- compute side ----
    auto load_q = [&](uint32_t (&qa)[Gm::KD][4], const SegIter& sg) {
        const uint16_t* qrow = p.q + ((size_t)sg.s * p.Hq + (size_t)sg.kvh * G) * D;
        const uint16_t* r0 = g < G ? qrow + g * D : nullptr;
        const uint16_t* r1 = (G > 8) ? qrow + (g + 8) * D : nullptr;
        if constexpr (Tr::KV8) {
            load_q_frags8<D>(qa, r0, r1, t4);
        } else {
            load_q_frags<D>(qa, r0, r1, t4);
        }
    };
    // the compute side's current chunk
    long long clo = 0, chi = 0;
    int cid = 0;
    SegIter it;
    auto pop_chunk = [&]() {
        __syncwarp();
        const ChunkEnt& e = cq[qhead % Tr::QN];
        clo = e.lo;
        chi = e.hi;
        cid = e.id;
        it.gi = e.lo;
        it.s = e.s;
        it.kvh = e.kvh;
        it.b0 = e.b0;
        it.nb = tab.nb(it.s);
        it.first = tab.fst(it.s);
        ++qhead;
    };
    pop_chunk();
    typename Tr::Acc acc;
    uint32_t qa[Gm::KD][4];
    load_q(qa, it);
    float qc[Tr::NR][2];   // 4-bit cache: the code offset per head (prepare_q4)
    auto q_to_f16 = [&]() {
        if constexpr (Tr::KV8) {
            if (__any_sync(0xffffffffu, q_frags8_to_f16<D, Tr::BF16>(qa)) && lane == 0)
                set_err(p.err, PA_DEVERR_Q_RANGE);
        }
        if constexpr (Tr::I4) prepare_q4<Gm::KD, Tr::NR>(qa, qc, lane);
    };
    q_to_f16();
    int ctx = tab.ctx[it.s];
    // The running state starts empty, or -- for the first suffix segment of
    // a sequence whose shared prefix was reduced by the prefix pass -- as the
    // prefix state (the carry), so the carry is folded in exactly once.
    auto init_acc = [&]() {
        acc.reset();
        if (it.first > 0 && it.b0 == 0) {
            const float* crow = p.carry + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * Tr::CSTRIDE;
            if constexpr (Tr::TR) {
                // heads 8 r + 2 t4 + c; the sum counted once (lanes g == 0)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int head = 8 * r + 2 * t4 + c;
                        if (head < G) {
                            acc.m[r][c] = __ldg(crow + head * Tr::CSTRIDE + D);
                            if (g == 0) acc.l[r][c] = __ldg(crow + head * Tr::CSTRIDE + D + 1);
                        }
                    }
            } else {
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r) {
                    const int head = g + 8 * r;
                    if (head < G) {
                        acc.m[r] = __ldg(crow + head * Tr::CSTRIDE + D);
                        if (t4 == 0) acc.l[r] = __ldg(crow + head * Tr::CSTRIDE + D + 1);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int head = 8 * r + 2 * t4 + (e & 1);
                        const int dim = 16 * mt + g + 8 * (e >> 1);
                        if (head < G) acc.o[mt][r][e] = __ldg(crow + head * Tr::CSTRIDE + dim);
                    }
        }
    };
    long long ncons = 0;      // stages folded in (or skipped after an abort)
    long long nwait = 0;      // stages whose copies are known to have landed
    int cst = 0;              // ring stage of the next stage to fold in (ncons % R)
    uint32_t cph = 0;         // and the parity of its fill ((ncons / R) & 1)
    const float qnan = __int_as_float(0x7fc00000);
    while (true) {
        const int len = seg_len(it, chi);
        // the next segment of this chunk: its position, length and Q fetched
        // a segment ahead
        SegIter nx = it;
        seg_advance(nx, len, p, tab);
        const bool nx_here = nx.gi < chi;
        uint32_t qn[Gm::KD][4];
        int ctx_next = 0;
        if (nx_here) {
            ctx_next = tab.ctx[nx.s];
            if constexpr (!Tr::KV8) load_q(qn, nx);   // the quantized paths keep the registers
        }
        init_acc();
        int poisoned = 0;
        for (int b = 0; b < len; b += UB) {
            const int st = cst;
            const uint32_t par = cph;
            if (++cst == R) {
                cst = 0;
                cph ^= 1u;
            }
            ++ncons;
            if (!aborted) {
                // every lane waits; the outcome is made warp-uniform
                const bool stall = p.stall_ns != 0 && ncons == 1;
                const bool ok = __all_sync(0xffffffffu, stall ? mbar_wait_bounded(stall_bar, 0, p.stall_ns)
                                                              : mbar_wait_bounded(full0 + 8 * st, par, p.timeout_ns));
                if (ok) {
                    nwait = ncons;
                } else {
                    if (lane == 0) set_err(p.err, PA_DEVERR_TIMEOUT);
                    aborted = true;
                }
            }
            if (aborted) {
                poisoned = 1;
                issue();
                continue;
            }
            poisoned |= stage_poison[st];
            const int nblk = min(UB, len - b);
            const int valid = min(nblk * BS, ctx - (it.first + it.b0 + b) * BS);
            const uint32_t kb = ring + st * Gm::STAGE_BYTES;
            bool zeroed = false;
            if constexpr (Tr::I4) {
                consume_stage4t<Gm, Tr::NR>(kb, valid, qa, qc, acc, p.scale_log2, lane);
            } else if constexpr (Tr::KV8) {
                consume_stage8t<Gm, Tr::NR, Tr::E5M2>(kb, valid, qa, acc, p.scale_log2, lane);
            } else {
                const uint32_t vb = kb + Gm::CHUNK_BYTES;
                if (valid < BS) {
                    zero_v_tail<Gm>(vb, valid, lane);
                    __syncwarp();
                    zeroed = true;
                }
                consume_block<Gm, Tr::NR, Tr::BF16>(kb, vb, valid, qa, acc, p.scale_log2, lane);
            }
            // the stage's shared memory is read (and any zeroing written)
            // before the async proxy refills it
            if (zeroed) fence_proxy_async_smem();
            __syncwarp();
            issue();
        }

        // ---- finish the segment: output rows, or this chunk's piece ----
        if constexpr (Tr::I4) fix_o4<D, Tr::NR>(acc);
        if constexpr (Tr::TR) {
            // sums over the 8 lanes of a head column (rows g)
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    acc.l[r][c] += __shfl_xor_sync(0xffffffffu, acc.l[r][c], 4);
                    acc.l[r][c] += __shfl_xor_sync(0xffffffffu, acc.l[r][c], 8);
                    acc.l[r][c] += __shfl_xor_sync(0xffffffffu, acc.l[r][c], 16);
                }
        } else {
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r) {
                acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 1);
                acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 2);
            }
        }
        const long long P0 = it.gi - it.b0;           // flattened start of this pair
        const long long cfirst = sc.of(P0);
        const long long clast = sc.of(P0 + it.nb - 1);
        const bool complete = cfirst == clast;
        uint16_t* orow = p.out + ((size_t)it.s * p.Hq + (size_t)it.kvh * G) * D;
        if (complete) {
#pragma unroll
            for (int r = 0; r < Tr::NR; ++r) {
                // this lane's o columns are heads 8 r + 2 t4 and 8 r + 2 t4 + 1
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int head = 8 * r + 2 * t4 + c;
                    float L;
                    if constexpr (Tr::TR) {
                        L = acc.l[r][c];
                    } else {
                        L = __shfl_sync(0xffffffffu, acc.l[r], (2 * t4 + c) * 4);
                    }
                    if (head < G) {
                        const float inv = p.v_scale / L;
#pragma unroll
                        for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int dim = 16 * mt + g + 8 * hh;
                                const float O = poisoned ? qnan : acc.o[mt][r][2 * hh + c];
                                orow[head * D + dim] = f32_to_16<Tr::BF16>(O * inv);
                            }
                    }
                }
            }
        } else {
            const int slot = (it.gi == clo) ? 0 : 1;
            float* prow = p.partials + ((size_t)cid * 2 + slot) * G * Tr::PSTRIDE;
#pragma unroll
            for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int head = 8 * r + 2 * t4 + (e & 1);
                        const int dim = 16 * mt + g + 8 * (e >> 1);
                        if (head < G) prow[head * Tr::PSTRIDE + dim] = poisoned ? qnan : acc.o[mt][r][e];
                    }
            if constexpr (Tr::TR) {
                if (g == 0) {
#pragma unroll
                    for (int r = 0; r < Tr::NR; ++r)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int head = 8 * r + 2 * t4 + c;
                            if (head < G) {
                                prow[head * Tr::PSTRIDE + D] = acc.m[r][c];
                                prow[head * Tr::PSTRIDE + D + 1] = acc.l[r][c];
                            }
                        }
                }
            } else if (t4 == 0) {
#pragma unroll
                for (int r = 0; r < Tr::NR; ++r) {
                    const int head = g + 8 * r;
                    if (head < G) {
                        prow[head * Tr::PSTRIDE + D] = acc.m[r];
                        prow[head * Tr::PSTRIDE + D + 1] = acc.l[r];
                    }
                }
            }
        }

        if (nx_here) {
            it = nx;
            ctx = ctx_next;
            if constexpr (Tr::KV8) {
                load_q(qa, it);
            } else {
#pragma unroll
                for (int kk = 0; kk < Gm::KD; ++kk)
#pragma unroll
                    for (int i = 0; i < 4; ++i) qa[kk][i] = qn[kk][i];
            }
        } else {
            // the chunk is done; the next one (if any) was queued by the
            // issue side, which is always ahead
            if (qhead == qtail) break;
            pop_chunk();
            ctx = tab.ctx[it.s];
            load_q(qa, it);
        }
        q_to_f16();
    }

    // After a timeout, wait (bounded, at the full limit) for the copies still
    // in flight before the CTA's shared memory is released.  Fill k of a ring
    // stage is issued only after fill k - R was waited for, so the fills not
    // known to have landed are the last R at most.
    if (aborted && lane == 0) {
        for (long long k = nwait; k < nreal; ++k) {
            if (k < nreal - R) continue;   // an older fill of the same stage
            mbar_wait_bounded(full0 + 8 * (uint32_t)(k % R), (uint32_t)((k / R) & 1), p.timeout_ns);
        }
    }
}

// Post-pass: for every pair cut by chunk boundaries, combine its pieces (in
// chunk order) by the log-sum-exp rule and write the output rows (a prefix
// carry is already inside the pair's first piece).  One warp per (pair, query head) -- two heads per warp when
// d = 64 -- so the whole merge is a few rounds of independent loads: first
// the lanes take different pieces to form the common max M and the sum L,
// then every lane folds 4 dims of every piece.  nworkers and nd are the
// decode launch's.
template <int D>
__global__ void __launch_bounds__(256, 4)
pa_decode_merge(const long long* __restrict__ cum, const float* __restrict__ partials, uint16_t* __restrict__ out,
                int N, int Hkv, int G, long long nworkers, int nd, float v_scale, int bf16) {
    griddep_wait();   // the decode grid is complete and its writes visible
    constexpr int PSTRIDE = D + 4;
    constexpr int LPH = D / 4;                     // lanes per head
    constexpr int HPW = 32 / LPH;                  // heads per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPH;
    const int hgroups = (G + HPW - 1) / HPW;
    const long long task = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const long long pair = task / hgroups;
    if (pair >= (long long)N * Hkv) return;
    const int s = (int)(pair / Hkv), kvh = (int)(pair % Hkv);
    const long long c0 = cum[s];
    const int nb = (int)(cum[s + 1] - c0);
    if (nb == 0) return;
    const Sched sc = make_sched(cum[N] * Hkv, nworkers, nd);
    const long long P0 = c0 * Hkv + (long long)kvh * nb;
    const long long cfirst = sc.of(P0), clast = sc.of(P0 + nb - 1);
    if (cfirst == clast) return;                                  // written by the decode kernel
    const int head0 = (int)(task % hgroups) * HPW + lane / LPH;
    const bool writer = head0 < G;
    const int head = writer ? head0 : G - 1;
    const int np = (int)(clast - cfirst) + 1;
    // piece i = chunk cfirst + i; only the first can sit in slot 1 (when the
    // pair starts inside that chunk)
    const size_t cstride = (size_t)2 * G * PSTRIDE;
    const float* first = partials + (size_t)cfirst * cstride + (sc.lo(cfirst) < P0 ? (size_t)G * PSTRIDE : 0) +
                         (size_t)head * PSTRIDE;
    const float* rest = partials + (size_t)cfirst * cstride + (size_t)head * PSTRIDE;
    auto piece = [&](int i) -> const float* { return i == 0 ? first : rest + (size_t)i * cstride; };
    const int Hq = Hkv * G;

    const int d0 = sub * 4;
    // the first pieces' o slices, issued before anything that depends on M
    constexpr int PB = 8;
    float4 v[PB];
#pragma unroll
    for (int k = 0; k < PB; ++k)
        if (k < np) v[k] = *reinterpret_cast<const float4*>(piece(k) + d0);
    // per-piece m and l: lane (i mod LPH) of the head's lane group holds piece i
    float M = -INFINITY;
    for (int i = sub; i < np; i += LPH) M = fmaxf(M, piece(i)[D]);
    for (int o = LPH / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float fi = sub < np ? ex2(piece(sub)[D] - M) : 0.f;   // factor of piece sub (np <= LPH)
    float L = 0.f;
    for (int i = sub; i < np; i += LPH) {
        const float* pr = piece(i);
        L += pr[D + 1] * ex2(pr[D] - M);
    }
    for (int o = LPH / 2; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int gbase = lane - sub;                                 // first lane of this head's group
    for (int c0 = 0; c0 < np; c0 += PB) {
        if (c0 > 0) {
#pragma unroll
            for (int k = 0; k < PB; ++k)
                if (c0 + k < np) v[k] = *reinterpret_cast<const float4*>(piece(c0 + k) + d0);
        }
#pragma unroll
        for (int k = 0; k < PB; ++k) {
            const int c = c0 + k;
            if (c >= np) break;
            const float f = c < LPH ? __shfl_sync(0xffffffffu, fi, gbase + c) : ex2(piece(c)[D] - M);
            acc.x += v[k].x * f;
            acc.y += v[k].y * f;
            acc.z += v[k].z * f;
            acc.w += v[k].w * f;
        }
    }
    if (!writer) return;
    const float inv = v_scale / L;
    const float x[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint16_t h0 = bf16 ? f32_to_16<true>(x[2 * k]) : f32_to_16<false>(x[2 * k]);
        const uint16_t h1 = bf16 ? f32_to_16<true>(x[2 * k + 1]) : f32_to_16<false>(x[2 * k + 1]);
        w[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
    }
    *reinterpret_cast<uint2*>(out + ((size_t)s * Hq + (size_t)kvh * G + head) * D + d0) = make_uint2(w[0], w[1]);
}

// ---------------------------------------------------------------- host side
struct DecodeLaunch {
    const CUtensorMap* tmap_k;
    const CUtensorMap* tmap_v;
    DecodeParams p;
    cudaStream_t stream;
    int grid;
    bool bf16;   // output type of the merge post-pass
};

struct DecodeKernelInfo {
    cudaError_t (*launch)(const DecodeLaunch&);
    int (*max_ctas)(int device);   // persistent grid size on that device, <= 0 on error
    int smem_bytes;
    int workers;                   // worker warps per CTA (partial-state slots per CTA)
};

template <class Tr>
cudaError_t decode_launch(const DecodeLaunch& L) {
    // launched with programmatic stream serialization: the CTAs' set-up
    // overlaps the pre-pass, and the kernel waits for it (griddep_wait)
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(L.grid, Tr::THREADS, Tr::SMEM_BYTES, L.stream, attr);
    return cudaLaunchKernelEx(&cfg, pa_decode_kernel<Tr>, *L.tmap_k, *L.tmap_v, L.p);
}

template <class Tr>
DecodeKernelInfo decode_info() {
    return DecodeKernelInfo{&decode_launch<Tr>, &persistent_ctas<pa_decode_kernel<Tr>, Tr::THREADS, Tr::SMEM_BYTES>,
                            Tr::SMEM_BYTES, Tr::NW};
}

// Per-(dtype, head_dim) tables, defined in the instantiation units.
// Index: [bs == 32][log2(g)]; the 8-bit tables add [e5m2] in front.
void decode8_table_bf16(DecodeKernelInfo (&t)[2][2][5]);
void decode8_table_fp16(DecodeKernelInfo (&t)[2][2][5]);
// 4-bit cache: [bs == 32][log2(g)]
void decode4_table_bf16(DecodeKernelInfo (&t)[2][5]);
void decode4_table_fp16(DecodeKernelInfo (&t)[2][5]);
void decode_table_bf16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_bf16_d64(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d128(DecodeKernelInfo (&t)[2][5]);
void decode_table_fp16_d64(DecodeKernelInfo (&t)[2][5]);

}  // namespace pa
