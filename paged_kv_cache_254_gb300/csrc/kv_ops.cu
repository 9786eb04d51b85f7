// KV-cache writes: appending new tokens' K/V at their slots, and copying whole
// blocks for copy-on-write.  Both move raw 16-byte vectors, so results are
// bit-exact.
//
// Append: token i goes to block slot / B, offset slot % B, for every KV head
// (thewebvale "vLLM & High-Throughput Serving", section 2, block table; ontq
// "AI Inference Serving at Scale", section 3, on-demand allocation).
// Copy: the block that a sharing sequence diverges in is cloned as a whole
// (ontq section 3, "Copy-on-Write Memory Sharing"; thewebvale section 2).
#include <cuda_runtime.h>
#include <cstdint>

#include "kv_ops.cuh"
#include "ptx.cuh"
#include "../../include/pa.h"
#include <cuda_fp16.h>

namespace pa {

// One thread per 16-byte vector of one (token, KV head) row.
__global__ void __launch_bounds__(256)
pa_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 const int64_t* __restrict__ slots, uint4* __restrict__ k_pool,
                 uint4* __restrict__ v_pool, AppendArgs a) {
    const long long total = (long long)a.T * a.Hkv * a.vec_per_row;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int vec = (int)(idx % a.vec_per_row);
        const long long rest = idx / a.vec_per_row;
        const int h = (int)(rest % a.Hkv);
        const long long i = rest / a.Hkv;
        const long long slot = __ldg(slots + i);
        if (slot < 0) continue;
        if (slot >= a.num_slots) {
            if (h == 0 && vec == 0 && a.err) atomicOr(a.err, PA_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / a.BS;
        const long long off = slot - blk * a.BS;
        const long long dst = ((blk * a.Hkv + h) * a.BS + off) * a.vec_per_row + vec;
        const long long src = (i * a.Hkv + h) * a.vec_per_row + vec;
        k_pool[dst] = __ldg(k_new + src);
        v_pool[dst] = __ldg(v_new + src);
    }
}

// blockIdx.y walks the pairs; the x dimension strides over the block's vectors.
__global__ void __launch_bounds__(256)
pa_copy_kernel(const int32_t* __restrict__ pairs, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
               CopyArgs a) {
    for (long long pi = blockIdx.y; pi < a.n; pi += gridDim.y) {
        const int src = __ldg(pairs + 2 * pi);
        const int dst = __ldg(pairs + 2 * pi + 1);
        if ((unsigned)src >= (unsigned)a.NB || (unsigned)dst >= (unsigned)a.NB) {
            if (blockIdx.x == 0 && threadIdx.x == 0 && a.err) atomicOr(a.err, PA_DEVERR_COPY_PAIR);
            continue;
        }
        if (src == dst) continue;
        const uint4* ks = k_pool + (long long)src * a.vec_per_block;
        uint4* kd = k_pool + (long long)dst * a.vec_per_block;
        const long long step = (long long)gridDim.x * blockDim.x;
        long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
        if (v_pool == nullptr) {   // a single pool (the 8-bit cache)
            for (; v < a.vec_per_block; v += step) kd[v] = ks[v];
            continue;
        }
        const uint4* vs = v_pool + (long long)src * a.vec_per_block;
        uint4* vd = v_pool + (long long)dst * a.vec_per_block;
        // four vectors of K and four of V in flight per thread
        for (; v + 3 * step < a.vec_per_block; v += 4 * step) {
            uint4 k0 = ks[v], k1 = ks[v + step], k2 = ks[v + 2 * step], k3 = ks[v + 3 * step];
            uint4 v0 = vs[v], v1 = vs[v + step], v2 = vs[v + 2 * step], v3 = vs[v + 3 * step];
            kd[v] = k0; kd[v + step] = k1; kd[v + 2 * step] = k2; kd[v + 3 * step] = k3;
            vd[v] = v0; vd[v + step] = v1; vd[v + 2 * step] = v2; vd[v + 3 * step] = v3;
        }
        for (; v < a.vec_per_block; v += step) {
            kd[v] = ks[v];
            vd[v] = vs[v];
        }
    }
}

// Quantising append for the 8-bit cache.  One thread per 16 head dims of one
// (token, KV head) row: each 16-bit value is divided by the cache scale in
// fp32 (round to nearest) and rounded to the nearest 8-bit code (ties to
// even, saturating).  Each (block, head) piece of the pool holds BS K rows
// of D bytes (16-byte parts permuted by XOR with the row index mod 8) and
// then the dims-first V ([D][BS] bytes).
template <bool BF16, bool E5M2>
__global__ void __launch_bounds__(256)
pa_append8_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                  const int64_t* __restrict__ slots, uint8_t* __restrict__ kv_pool, Append8Args a) {
    const int groups = a.D / 16;
    const long long total = (long long)a.T * a.Hkv * groups;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int grp = (int)(idx % groups);
        const long long rest = idx / groups;
        const int h = (int)(rest % a.Hkv);
        const long long i = rest / a.Hkv;
        const long long slot = __ldg(slots + i);
        if (slot < 0) continue;
        if (slot >= a.num_slots) {
            if (h == 0 && grp == 0 && a.err) atomicOr(a.err, PA_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / a.BS;
        const int off = (int)(slot - blk * a.BS);
        const long long src = (i * a.Hkv + h) * a.D + 16 * grp;
        auto widen = [](uint16_t x) -> float {
            if constexpr (BF16) return __uint_as_float((uint32_t)x << 16);
            return __half2float(__ushort_as_half(x));
        };
        uint16_t kv[16], vv[16];
        {
            const uint4 k0 = __ldg(reinterpret_cast<const uint4*>(k_new + src));
            const uint4 k1 = __ldg(reinterpret_cast<const uint4*>(k_new + src + 8));
            const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(v_new + src));
            const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(v_new + src + 8));
            const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
            const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                kv[2 * j] = (uint16_t)(kw[j] & 0xffffu);
                kv[2 * j + 1] = (uint16_t)(kw[j] >> 16);
                vv[2 * j] = (uint16_t)(vw[j] & 0xffffu);
                vv[2 * j + 1] = (uint16_t)(vw[j] >> 16);
            }
        }
        uint32_t kq[4];
        uint8_t vq[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint16_t kp = f32x2_to_fp8x2<E5M2>(__fdiv_rn(widen(kv[2 * j]), a.k_scale),
                                                     __fdiv_rn(widen(kv[2 * j + 1]), a.k_scale));
            const uint16_t vp = f32x2_to_fp8x2<E5M2>(__fdiv_rn(widen(vv[2 * j]), a.v_scale),
                                                     __fdiv_rn(widen(vv[2 * j + 1]), a.v_scale));
            if (j & 1) kq[j >> 1] |= (uint32_t)kp << 16; else kq[j >> 1] = kp;
            vq[2 * j] = (uint8_t)(vp & 0xffu);
            vq[2 * j + 1] = (uint8_t)(vp >> 8);
        }
        uint8_t* piece = kv_pool + (blk * a.Hkv + h) * 2 * a.BS * a.D;
        // K row `off`: 16-byte part grp stored at part position grp ^ (off % 8)
        uint8_t* kdst = piece + (long long)off * a.D + 16 * (grp ^ (off & 7));
        *reinterpret_cast<uint4*>(kdst) = make_uint4(kq[0], kq[1], kq[2], kq[3]);
        uint8_t* vdst = piece + (long long)a.BS * a.D + (long long)(16 * grp) * a.BS + off;
#pragma unroll
        for (int j = 0; j < 16; ++j) vdst[(long long)j * a.BS] = vq[j];
    }
}

// Quantising append for the 4-bit cache (head_dim 128).  One warp per
// (token, KV head) row; lane L holds dims 4L .. 4L + 3.  Per row: scale =
// amax / 7 (fp32 division), code = rint(x / scale) clamped to [-8, 7] (0 for a
// zero row).  K codes fill whole 32-bit words of the token's row; V is stored
// dims-first, where neighbouring tokens share words, so each V nibble is set
// with an atomic AND (clear) and OR (set) that touch only its own bits.
template <bool BF16>
__global__ void __launch_bounds__(256)
pa_append4_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                  const int64_t* __restrict__ slots, uint8_t* __restrict__ kv_pool, Append4Args a) {
    constexpr int D = 128;
    const int lane = threadIdx.x & 31;
    const int BS = a.BS;
    const int VC = BS * 64, KS = BS * 128, VS = KS + 4 * BS;
    const long long rows = (long long)a.T * a.Hkv;
    const long long wstride = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < rows; w += wstride) {
        const long long i = w / a.Hkv;
        const int h = (int)(w - i * a.Hkv);
        const long long slot = __ldg(slots + i);
        if (slot < 0) continue;
        if (slot >= a.num_slots) {
            if (h == 0 && lane == 0 && a.err) atomicOr(a.err, PA_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / BS;
        const int off = (int)(slot - blk * BS);
        uint8_t* piece = kv_pool + (blk * a.Hkv + h) * (long long)a.piece_bytes;
        const long long src = (i * a.Hkv + h) * D + 4 * lane;
        auto widen = [](uint16_t x) -> float {
            if constexpr (BF16) return __uint_as_float((uint32_t)x << 16);
            return __half2float(__ushort_as_half(x));
        };
        const uint2 kw = __ldg(reinterpret_cast<const uint2*>(k_new + src));
        const uint2 vw = __ldg(reinterpret_cast<const uint2*>(v_new + src));
        float kx[4] = {widen(kw.x & 0xffffu), widen(kw.x >> 16), widen(kw.y & 0xffffu), widen(kw.y >> 16)};
        float vx[4] = {widen(vw.x & 0xffffu), widen(vw.x >> 16), widen(vw.y & 0xffffu), widen(vw.y >> 16)};
        float ka = 0.f, va = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ka = fmaxf(ka, fabsf(kx[e]));
            va = fmaxf(va, fabsf(vx[e]));
        }
        for (int o = 16; o > 0; o >>= 1) {
            ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, o));
            va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, o));
        }
        const float ks = __fdiv_rn(ka, 7.f), vs = __fdiv_rn(va, 7.f);
        auto code = [](float x, float s) -> uint32_t {
            if (!(s > 0.f)) return 8u;                       // code 0
            const float q = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -8.f), 7.f);
            return (uint32_t)((int)q + 8);
        };
        auto nib = [](int e) -> int { return (e & 1) ? 4 + (e >> 1) : (e >> 1); };
        // K: word lane / 2 of the token's row holds dims 8 (lane / 2) .. + 7
        uint32_t part = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) part |= code(kx[e], ks) << (4 * nib(4 * (lane & 1) + e));
        part |= __shfl_xor_sync(0xffffffffu, part, 1);
        if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(piece + off * 64 + 4 * (lane >> 1)) = part;
        // V: dims-first rows of BS nibbles; this token is element off % 8 of word off / 8
        const int pos = 4 * nib(off & 7);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            unsigned int* wp = reinterpret_cast<unsigned int*>(piece + VC + (4 * lane + e) * (BS / 2) + 4 * (off >> 3));
            atomicAnd(wp, ~(0xfu << pos));
            atomicOr(wp, code(vx[e], vs) << pos);
        }
        if (lane == 0) {
            *reinterpret_cast<float*>(piece + KS + 4 * off) = ks;
            *reinterpret_cast<float*>(piece + VS + 4 * off) = vs;
        }
    }
}

cudaError_t append4_launch(const void* k_new, const void* v_new, const int64_t* slots, void* kv_pool,
                           const Append4Args& a, bool bf16, cudaStream_t stream, int sms) {
    const long long rows = (long long)a.T * a.Hkv;
    long long blocks = (rows + 7) / 8;                    // 8 warps per CTA
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto kn = static_cast<const uint16_t*>(k_new);
    auto vn = static_cast<const uint16_t*>(v_new);
    auto kv = static_cast<uint8_t*>(kv_pool);
    if (bf16) pa_append4_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
    else pa_append4_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
    return cudaGetLastError();
}

cudaError_t append8_launch(const void* k_new, const void* v_new, const int64_t* slots, void* kv_pool,
                           const Append8Args& a, bool bf16, bool e5m2, cudaStream_t stream, int sms) {
    const long long total = (long long)a.T * a.Hkv * (a.D / 16);
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto kn = static_cast<const uint16_t*>(k_new);
    auto vn = static_cast<const uint16_t*>(v_new);
    auto kv = static_cast<uint8_t*>(kv_pool);
    if (bf16) {
        if (e5m2) pa_append8_kernel<true, true><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
        else pa_append8_kernel<true, false><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
    } else {
        if (e5m2) pa_append8_kernel<false, true><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
        else pa_append8_kernel<false, false><<<(unsigned)blocks, 256, 0, stream>>>(kn, vn, slots, kv, a);
    }
    return cudaGetLastError();
}

cudaError_t append_launch(const void* k_new, const void* v_new, const int64_t* slots, void* k_pool,
                          void* v_pool, const AppendArgs& a, cudaStream_t stream, int sms) {
    const long long total = (long long)a.T * a.Hkv * a.vec_per_row;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    pa_append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots,
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), a);
    return cudaGetLastError();
}

cudaError_t copy_launch(const int32_t* pairs, void* k_pool, void* v_pool, const CopyArgs& a,
                        cudaStream_t stream, int sms) {
    // enough CTAs per pair to cover the block in one pass of 4 vectors per thread
    long long gx = (a.vec_per_block + 4 * 256 - 1) / (4 * 256);
    if (gx < 1) gx = 1;
    long long gy = a.n;
    const long long cap = (long long)sms * 16;
    if (gx * gy > cap) gy = cap / gx > 0 ? cap / gx : 1;
    if (gy > 65535) gy = 65535;
    pa_copy_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, stream>>>(
        pairs, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), a);
    return cudaGetLastError();
}

}  // namespace pa
