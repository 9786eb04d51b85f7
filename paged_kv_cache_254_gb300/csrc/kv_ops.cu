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
#include "../../include/pa.h"

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
        const uint4* vs = v_pool + (long long)src * a.vec_per_block;
        uint4* kd = k_pool + (long long)dst * a.vec_per_block;
        uint4* vd = v_pool + (long long)dst * a.vec_per_block;
        const long long step = (long long)gridDim.x * blockDim.x;
        long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
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
