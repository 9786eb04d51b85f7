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
