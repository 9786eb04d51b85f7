// Pieces shared by the paged decode kernels: block geometry, work-range
// arithmetic, and the per-warp update of one KV block (scores, online
// softmax, PV) on mma.sync fragments.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"
#include "../../include/pa.h"

namespace pa {

// Launch configuration with programmatic stream serialization: the kernel
// may start while the stream's previous kernel runs, and waits for it with
// griddepcontrol.wait before reading anything the stream wrote.  `attr`
// holds the attribute the configuration points to.
inline cudaLaunchConfig_t pdl_config(long long grid, int threads, int smem, cudaStream_t stream,
                                     cudaLaunchAttribute (&attr)[1]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// One (block, KV head) chunk of the 16-bit cache as it sits in a ring stage:
// HALVES boxes of BS rows x 128 bytes, 128-byte swizzled; the K chunk, then
// the V chunk.  One stage holds one block.
template <int D_, int BS_>
struct Geom {
    static constexpr int D = D_;
    static constexpr int BS = BS_;
    static constexpr int HALVES = D * 2 / 128;
    static constexpr int BOX_BYTES = BS * 128;
    static constexpr int CHUNK_BYTES = HALVES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int UB = 1;         // blocks per stage
    static constexpr int NT = BS / 8;    // 8-token n-tiles of S^T
    static constexpr int KT = BS / 16;   // 16-token k-steps of PV
    static constexpr int KD = D / 16;    // 16-dim k-steps of QK, m-tiles of PV
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
};

// The 8-bit cache (head_dim 128): a (block, KV head) piece is BS K rows of
// 128 bytes (16-byte parts of row r permuted by XOR with r % 8, so a plain
// copy lands them bank-spread) followed by the dims-first V (128 rows of BS
// bytes), one contiguous run of PIECE_BYTES in the pool.  A ring stage holds
// UB consecutive blocks of one (sequence, KV head) pair: 32 tokens.
template <int BS_>
struct Geom8 {
    static constexpr int D = 128;
    static constexpr int BS = BS_;
    static constexpr int PIECE_BYTES = 2 * BS * 128;
    static constexpr int UB = 32 / BS;
    // piece u of a stage sits at u * PIECE_PAD: with two pieces per stage the
    // second is moved by 64 bytes, so the V rows of both pieces that one load
    // instruction reads fall in different shared-memory banks
    static constexpr int PIECE_PAD = UB == 2 ? PIECE_BYTES + 64 : PIECE_BYTES;
    static constexpr int STAGE_BYTES = UB * PIECE_PAD;
    static constexpr int COPY_BYTES = UB * PIECE_BYTES;   // bytes copied into a full stage
    static constexpr int KD = D / 16;
    static constexpr int TOK = 32;                         // tokens per stage
    __host__ __device__ static constexpr int poff(int u) { return u * PIECE_PAD; }
    static_assert(BS == 16 || BS == 32, "block_size");
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

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

template <int BOX_BYTES>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)((chunk >> 3) * BOX_BYTES + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <bool BF16>
__device__ __forceinline__ uint16_t f32_to_16(float x) {
    uint16_t r;
    if constexpr (BF16) {
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    } else {
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
    }
    return r;
}

template <bool BF16>
__device__ __forceinline__ uint16_t qnan16() {
    return BF16 ? (uint16_t)0x7fc0 : (uint16_t)0x7e00;
}

// Running softmax state of one warp for up to 8 * NR query rows (fragment row
// g and, for NR == 2, row g + 8).  m is in the exp2 domain (scores already
// multiplied by scale * log2(e)); l and o are per-lane partial sums.
template <int D, int NR>
struct WarpAcc {
    float m[NR], l[NR];
    float o[D / 16][NR][4];   // O^T fragments: dims x rows

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][r][e] = 0.f;
    }
};

// A-operand fragments of Q (rows = query rows, k = head dims) for one warp.
// row0 / row1: the query row this lane's fragment rows g and g + 8 hold, or
// null for an unused (zero) row.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[D / 16][4], const uint16_t* row0,
                                             const uint16_t* row1, int t4) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = kk * 16 + 2 * t4;
        qa[kk][0] = row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + c)) : 0u;
        qa[kk][2] = row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + c + 8)) : 0u;
        qa[kk][1] = row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + c)) : 0u;
        qa[kk][3] = row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + c + 8)) : 0u;
    }
}

// Fold one KV block (K chunk at kb, V chunk at vb, shared-memory addresses)
// into the warp's state.  Tokens at offsets >= valid are masked out; when
// valid < BS the caller has made the V rows past `valid` finite (zero).
//   S^T = Q K^T        : mma rows = query rows, n = tokens, k = dims
//   online softmax     : row max over the 4 lanes of a fragment row
//   O^T += V^T P^T     : m = dims, n = query rows, k = tokens; P as hi + lo
template <class Gm, int NR, bool BF16>
__device__ __forceinline__ void consume_block(uint32_t kb, uint32_t vb, int valid,
                                              const uint32_t (&qa)[Gm::KD][4], WarpAcc<Gm::D, NR>& acc,
                                              float scale_log2, int lane) {
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
            const float v = tok < valid ? sacc[nt][e] * scale_log2 : -INFINITY;
            sacc[nt][e] = v;
            if ((e >> 1) < NR) mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
    float alpha[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(acc.m[r], mx[r]);
        alpha[r] = ex2(acc.m[r] - m_new);
        acc.m[r] = m_new;
        acc.l[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = e >> 1;
            if (r < NR) {
                const float pe = ex2(sacc[nt][e] - acc.m[r]);
                sacc[nt][e] = pe;
                acc.l[r] += pe;
            }
        }
    // P^T fragments (B operand of PV): k = tokens, n = rows.  P enters as
    // hi + lo, two 16-bit parts (hi = round(p), lo = round(p - hi)), keeping
    // ~16 bits of p instead of the 8 a single bf16 would leave.
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

    // rescale the running O^T by exp2(m_old - m_new) of each row; skipped
    // (a multiplication by exactly 1) when no row's maximum moved
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        if (__any_sync(0xffffffffu, alpha[r] != 1.f)) {
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
    }

#pragma unroll
    for (int mt = 0; mt < Gm::KD; ++mt)
#pragma unroll
        for (int kt = 0; kt < Gm::KT; ++kt) {
            uint32_t a0, a1, a2, a3;
            const int row = kt * 16 + ((lane >> 4) << 3) + (lane & 7);
            const int chunk = 2 * mt + ((lane >> 3) & 1);
            ldsm_x4_t(vb + swz<Gm::BOX_BYTES>(row, chunk), a0, a1, a2, a3);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                mma16816<BF16>(acc.o[mt][r], a0, a1, a2, a3, pb[kt][r][0], pb[kt][r][1]);
                mma16816<BF16>(acc.o[mt][r], a0, a1, a2, a3, pl[kt][r][0], pl[kt][r][1]);
            }
        }
}

// ---------------------------------------------------------------- 8-bit cache
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Q fragments for the 8-bit path with the head dims in the order the K bytes
// are read: k-step kk, fragment column 2 t4 + e -> dim 32 t4 + 4 kk + e,
// column 2 t4 + 8 + e -> dim 32 t4 + 4 kk + 2 + e.  Loaded as stored (q's
// 16-bit type); q_frags8_to_f16 then turns bf16 pairs into fp16 pairs.
template <int D>
__device__ __forceinline__ void load_q_frags8(uint32_t (&qa)[D / 16][4], const uint16_t* row0,
                                              const uint16_t* row1, int t4) {
    auto ld = [](const uint16_t* p) -> uint32_t { return __ldg(reinterpret_cast<const uint32_t*>(p)); };
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = 32 * t4 + 4 * kk;
        qa[kk][0] = row0 ? ld(row0 + c) : 0u;
        qa[kk][2] = row0 ? ld(row0 + c + 2) : 0u;
        qa[kk][1] = row1 ? ld(row1 + c) : 0u;
        qa[kk][3] = row1 ? ld(row1 + c + 2) : 0u;
    }
}

// Returns true on this lane if an element left fp16's finite range (a bf16
// query beyond 65504, or a non-finite one).
template <int D, bool QBF16>
__device__ __forceinline__ bool q_frags8_to_f16(uint32_t (&qa)[D / 16][4]) {
    bool bad = false;
    if constexpr (QBF16) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t h = bf16x2_to_f16x2(qa[kk][i]);
                bad |= (h & 0x7c00u) == 0x7c00u || (h & 0x7c000000u) == 0x7c000000u;
                qa[kk][i] = h;
            }
    }
    return bad;
}

// The 4-bit cache (head_dim 128): a (block, KV head) piece is the K codes
// token-major (BS rows of 64 bytes), the V codes dims-first (128 rows of
// BS / 2 bytes), then BS fp32 K scales and BS fp32 V scales -- one
// contiguous run of PIECE_BYTES in the pool.  Codes are nibbles code + 8; in
// each 32-bit word of 8 elements, element 2k sits in nibble k and element
// 2k + 1 in nibble k + 4.  A ring stage holds UB blocks of one pair: 64 tokens.
template <int BS_>
struct Geom4 {
    static constexpr int D = 128;
    static constexpr int BS = BS_;
    static constexpr int VC = BS * 64;                 // V codes offset
    static constexpr int KS = BS * 128;                // K scales offset
    static constexpr int VS = KS + 4 * BS;             // V scales offset
    static constexpr int PIECE_BYTES = VS + 4 * BS;
    // a stage is 64 tokens: two halves of 32, each read like an 8-bit stage
    static constexpr int TOK = 64;
    static constexpr int UB = TOK / BS;
    // piece u at poff(u): with 16-token blocks 64 bytes of padding follow
    // every even piece, so the two pieces of a half start 64 bytes apart
    // modulo 128 and sit in different shared-memory banks
    __host__ __device__ static constexpr int poff(int u) {
        return u * PIECE_BYTES + (BS == 16 ? 64 * ((u + 1) >> 1) : 0);
    }
    static_assert(BS == 32 || (PIECE_BYTES % 128 == 0 && (poff(1) - poff(0)) % 128 == 64 &&
                               (poff(3) - poff(2)) % 128 == 64 && poff(2) >= poff(1) + PIECE_BYTES),
                  "pieces of a stage must not overlap, and the two of a half must differ by 64 modulo 128");
    static constexpr int STAGE_BYTES = poff(UB - 1) + PIECE_BYTES;
    static constexpr int COPY_BYTES = UB * PIECE_BYTES;
    static constexpr int KD = D / 16;
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(PIECE_BYTES % 16 == 0, "pieces are copied in 16-byte units");
};

// Zero the V rows at offsets >= valid of a partly filled block (they may hold
// anything, NaN included, and 0 * NaN would poison the PV product).
template <class Gm>
__device__ __forceinline__ void zero_v_tail(uint32_t vb, int valid, int lane) {
    const int nz = (Gm::BS - valid) * Gm::HALVES * 8;   // 16-byte pieces
    for (int i = lane; i < nz; i += 32) {
        const int piece = i & 7;
        const int rest = i >> 3;
        const int h = rest % Gm::HALVES;
        const int row = valid + rest / Gm::HALVES;
        const uint32_t a = vb + h * Gm::BOX_BYTES + row * 128 + piece * 16;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(a), "r"(0) : "memory");
    }
}

// Combine a state (m2, l2, o2) into (M, L, O) by the log-sum-exp rule.
__device__ __forceinline__ void lse_fold(float& M, float& L, float& O, float m2, float l2, float o2) {
    const float Mn = fmaxf(M, m2);
    const float fa = ex2(M - Mn), fb = ex2(m2 - Mn);
    L = L * fa + l2 * fb;
    O = O * fa + o2 * fb;
    M = Mn;
}

// Persistent grid size: SMs x resident CTAs of `Kernel` (cached per device).
template <auto Kernel, int THREADS, int SMEM>
int persistent_ctas(int device) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return -1;
    if (cached[device] > 0) return cached[device];
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return -1;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return -1;
    int sms = 0, per_sm = 0;
    cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, Kernel, THREADS, SMEM);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || per_sm <= 0) return -1;
    cached[device] = sms * per_sm;
    return cached[device];
}

}  // namespace pa
