// C ABI of libpa (declared in include/pa.h): host-side argument checks,
// kernel selection, TMA descriptor set-up and launches.  Nothing here
// allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/pa.h"
#include "decode_kernel.cuh"
#include "kv_ops.cuh"
#include "prefix_kernel.cuh"

namespace {

using namespace pa;

constexpr uint64_t kTimeoutNs = 2000000000ull;   // bound on any device-side wait

struct DecodeTables {
    DecodeKernelInfo t[2][2][2][5];   // [bf16][d == 128][bs == 32][log2 g]
};

const DecodeTables& decode_tables() {
    static const DecodeTables tabs = [] {
        DecodeTables d;
        decode_table_fp16_d64(d.t[0][0]);
        decode_table_fp16_d128(d.t[0][1]);
        decode_table_bf16_d64(d.t[1][0]);
        decode_table_bf16_d128(d.t[1][1]);
        return d;
    }();
    return tabs;
}

int log2_exact(int g) {
    switch (g) {
        case 1: return 0;
        case 2: return 1;
        case 4: return 2;
        case 8: return 3;
        case 16: return 4;
        default: return -1;
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int elem_bytes(int dtype) {
    switch (dtype) {
        case PA_FP16:
        case PA_BF16: return 2;
        case PA_FP8_E4M3:
        case PA_FP8_E5M2: return 1;
        default: return 0;
    }
}

// Checks shared by all entry points (fields every call uses).
pa_status check_common(const pa_shape* s) {
    if (!s) return PA_ERR_INVALID_ARG;
    if (s->num_kv_heads <= 0 || s->head_dim <= 0 || s->block_size <= 0 || s->num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (elem_bytes(s->dtype) == 0) return PA_ERR_INVALID_ARG;
    if ((s->head_dim * elem_bytes(s->dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;   // 16-byte rows
    if ((long long)s->num_blocks * s->num_kv_heads * s->block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

pa_status pick_decode(const pa_shape* s, const DecodeKernelInfo** out) {
    pa_status st = check_common(s);
    if (st != PA_OK) return st;
    if (s->dtype != PA_FP16 && s->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (s->num_seqs < 0 || s->num_q_heads <= 0 || s->max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (s->num_q_heads % s->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if ((long long)s->max_blocks_per_seq * s->block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    const int lg = log2_exact(s->num_q_heads / s->num_kv_heads);
    if (lg < 0) return PA_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (s->block_size != 16 && s->block_size != 32) return PA_ERR_UNSUPPORTED;
    *out = &decode_tables().t[s->dtype == PA_BF16][s->head_dim == 128][s->block_size == 32][lg];
    return PA_OK;
}

size_t counters_bytes(const pa_shape* s) {
    const size_t c = (size_t)s->num_seqs * s->num_kv_heads * sizeof(int32_t);
    return (c + 255) & ~size_t(255);
}

size_t partials_bytes(const pa_shape* s, int max_ctas) {
    const int g = s->num_q_heads / s->num_kv_heads;
    return (size_t)max_ctas * 2 * g * (s->head_dim + 2) * sizeof(float);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The pool viewed as a 2-D tensor: rows = (block, kv head, slot), columns =
// head_dim; boxes of 64 columns x block_size rows land 128-byte swizzled.
bool pool_map(CUtensorMap* m, const void* pool, const pa_shape* s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)s->head_dim,
                                (cuuint64_t)s->num_blocks * s->num_kv_heads * s->block_size};
    const cuuint64_t strides[1] = {(cuuint64_t)s->head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)s->block_size};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 2, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}


const DecodeKernelInfo* pick_decode8(const pa_shape* s, int kv_format) {
    static const auto tab = [] {
        struct T { DecodeKernelInfo bf[2][2][5], fp[2][2][5]; } x;
        decode8_table_bf16(x.bf);
        decode8_table_fp16(x.fp);
        return x;
    }();
    const int lg = log2_exact(s->num_q_heads / s->num_kv_heads);
    const int f = kv_format == PA_FP8_E5M2 ? 1 : 0;
    const int b = s->block_size == 32 ? 1 : 0;
    return s->dtype == PA_BF16 ? &tab.bf[f][b][lg] : &tab.fp[f][b][lg];
}

pa_status check_fp8(const pa_shape* s, int kv_format, float k_scale, float v_scale) {
    if (kv_format != PA_FP8_E4M3 && kv_format != PA_FP8_E5M2) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (s->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if ((long long)s->num_blocks * s->num_kv_heads * s->block_size * 2 >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

const PrefixKernelInfo& pick_prefix(const pa_shape* s) {
    static const auto tab = [] {
        struct T { PrefixKernelInfo t[2][2][2]; } x;
        prefix_table(x.t);
        return x;
    }();
    return tab.t[s->dtype == PA_BF16][s->head_dim == 128][s->block_size == 32];
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of prefix-aware decode: decode counters, prefix counters, carry
// states, decode partials, prefix partials (offsets in off[0..4]).
size_t shared_prefix_layout(const pa_shape* s, int dec_ctas, int pre_ctas, size_t (&off)[6]) {
    const size_t cb = counters_bytes(s);
    off[0] = 0;                                   // decode counters
    off[1] = cb;                                  // prefix counters
    off[5] = 2 * cb;                              // first block per sequence
    off[2] = off[5] + align256((size_t)s->num_seqs * sizeof(int32_t));   // carry (after the zeroed part)
    const size_t carry = align256((size_t)s->num_seqs * s->num_q_heads * (s->head_dim + 2) * sizeof(float));
    off[3] = off[2] + carry;
    off[4] = off[3] + align256(partials_bytes(s, dec_ctas));
    return off[4] + (size_t)pre_ctas * 2 * 32 * (s->head_dim + 2) * sizeof(float);
}

}  // namespace

extern "C" {

size_t pa_decode_workspace_bytes(const pa_shape* shape) {
    const DecodeKernelInfo* k = nullptr;
    if (pick_decode(shape, &k) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return 0;
    return counters_bytes(shape) + partials_bytes(shape, ctas);
}

pa_status pa_decode(const pa_shape* shape, const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                    void* workspace, size_t workspace_bytes, uint32_t* err_word, void* stream) {
    const DecodeKernelInfo* k = nullptr;
    pa_status st = pick_decode(shape, &k);
    if (st != PA_OK) return st;
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->num_seqs == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return PA_ERR_CUDA;
    const size_t need = counters_bytes(shape) + partials_bytes(shape, ctas);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!pool_map(&mk, k_pool, shape) || !pool_map(&mv, v_pool, shape)) return PA_ERR_CUDA;

    DecodeLaunch L{};
    L.tmap_k = &mk;
    L.tmap_v = &mv;
    L.p.q = static_cast<const uint16_t*>(q);
    L.p.block_tables = block_tables;
    L.p.context_lens = context_lens;
    L.p.out = static_cast<uint16_t*>(out);
    L.p.counters = static_cast<int32_t*>(workspace);
    L.p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counters_bytes(shape));
    L.p.err = err_word;
    L.p.N = shape->num_seqs;
    L.p.Hq = shape->num_q_heads;
    L.p.Hkv = shape->num_kv_heads;
    L.p.NB = shape->num_blocks;
    L.p.MB = shape->max_blocks_per_seq;
    L.p.scale_log2 = (float)((double)scale * 1.4426950408889634);   // log2(e)
    L.p.timeout_ns = kTimeoutNs;
    L.p.v_scale = 1.0f;
    L.stream = static_cast<cudaStream_t>(stream);
    L.grid = ctas;
    // Arrival counters start at zero for every call (the region may hold
    // another shape's partial states from an earlier call).
    if (cudaMemsetAsync(workspace, 0, counters_bytes(shape), L.stream) != cudaSuccess) return PA_ERR_CUDA;
    return k->launch(L) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_shared_prefix_workspace_bytes(const pa_shape* shape) {
    const DecodeKernelInfo* k = nullptr;
    if (pick_decode(shape, &k) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int dec = k->max_ctas(dev), pre = pick_prefix(shape).max_ctas(dev);
    if (dec <= 0 || pre <= 0) return 0;
    size_t off[6];
    return shared_prefix_layout(shape, dec, pre, off);
}

pa_status pa_decode_shared_prefix(const pa_shape* shape, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const int32_t* context_lens, int32_t num_groups,
                                  const int32_t* group_starts, const int32_t* group_prefix_blocks, float scale,
                                  void* out, void* workspace, size_t workspace_bytes, uint32_t* err_word,
                                  void* stream) {
    const DecodeKernelInfo* k = nullptr;
    pa_status st = pick_decode(shape, &k);
    if (st != PA_OK) return st;
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || num_groups < 0) return PA_ERR_INVALID_ARG;
    if (num_groups > 0 && (!group_starts || !group_prefix_blocks || !aligned(group_starts, 4) ||
                           !aligned(group_prefix_blocks, 4)))
        return PA_ERR_INVALID_ARG;
    if (shape->num_seqs == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const PrefixKernelInfo& pk = pick_prefix(shape);
    const int dec = k->max_ctas(dev), pre = pk.max_ctas(dev);
    if (dec <= 0 || pre <= 0) return PA_ERR_CUDA;
    size_t off[6];
    const size_t need = shared_prefix_layout(shape, dec, pre, off);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!pool_map(&mk, k_pool, shape) || !pool_map(&mv, v_pool, shape)) return PA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    const float scale_log2 = (float)((double)scale * 1.4426950408889634);   // log2(e)
    // both arrival-counter regions and the first-block array start at zero
    if (cudaMemsetAsync(ws, 0, off[2], strm) != cudaSuccess) return PA_ERR_CUDA;

    if (num_groups > 0) {
        PrefixLaunch P{};
        P.tmap_k = &mk;
        P.tmap_v = &mv;
        P.p.q = static_cast<const uint16_t*>(q);
        P.p.block_tables = block_tables;
        P.p.context_lens = context_lens;
        P.p.grp_starts = group_starts;
        P.p.grp_prefix = group_prefix_blocks;
        P.p.carry = reinterpret_cast<float*>(ws + off[2]);
        P.p.first_blocks = reinterpret_cast<int32_t*>(ws + off[5]);
        P.p.counters = reinterpret_cast<int32_t*>(ws + off[1]);
        P.p.partials = reinterpret_cast<float*>(ws + off[4]);
        P.p.err = err_word;
        P.p.n_groups = num_groups;
        P.p.G = shape->num_q_heads / shape->num_kv_heads;
        P.p.N = shape->num_seqs;
        P.p.Hq = shape->num_q_heads;
        P.p.Hkv = shape->num_kv_heads;
        P.p.NB = shape->num_blocks;
        P.p.MB = shape->max_blocks_per_seq;
        P.p.scale_log2 = scale_log2;
        P.p.timeout_ns = kTimeoutNs;
        P.stream = strm;
        P.grid = pre;
        if (pk.launch(P) != cudaSuccess) return PA_ERR_CUDA;
    }

    DecodeLaunch L{};
    L.tmap_k = &mk;
    L.tmap_v = &mv;
    L.p.q = static_cast<const uint16_t*>(q);
    L.p.block_tables = block_tables;
    L.p.context_lens = context_lens;
    L.p.out = static_cast<uint16_t*>(out);
    L.p.counters = reinterpret_cast<int32_t*>(ws + off[0]);
    L.p.partials = reinterpret_cast<float*>(ws + off[3]);
    L.p.err = err_word;
    L.p.first_blocks = reinterpret_cast<const int32_t*>(ws + off[5]);
    L.p.carry = reinterpret_cast<const float*>(ws + off[2]);
    L.p.N = shape->num_seqs;
    L.p.Hq = shape->num_q_heads;
    L.p.Hkv = shape->num_kv_heads;
    L.p.NB = shape->num_blocks;
    L.p.MB = shape->max_blocks_per_seq;
    L.p.scale_log2 = scale_log2;
    L.p.timeout_ns = kTimeoutNs;
    L.p.v_scale = 1.0f;
    L.stream = strm;
    L.grid = dec;
    return k->launch(L) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_fp8_workspace_bytes(const pa_shape* shape, int32_t kv_format) {
    const DecodeKernelInfo* k16 = nullptr;
    if (pick_decode(shape, &k16) != PA_OK || check_fp8(shape, kv_format, 1.f, 1.f) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int ctas = pick_decode8(shape, kv_format)->max_ctas(dev);
    if (ctas <= 0) return 0;
    return counters_bytes(shape) + partials_bytes(shape, ctas);
}

pa_status pa_decode_fp8(const pa_shape* shape, int32_t kv_format, const void* q, const void* kv_pool,
                        const int32_t* block_tables, const int32_t* context_lens, float scale, float k_scale,
                        float v_scale, void* out, void* workspace, size_t workspace_bytes, uint32_t* err_word,
                        void* stream) {
    const DecodeKernelInfo* k16 = nullptr;
    pa_status st = pick_decode(shape, &k16);
    if (st != PA_OK) return st;
    st = check_fp8(shape, kv_format, k_scale, v_scale);
    if (st != PA_OK) return st;
    if (!q || !kv_pool || !block_tables || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->num_seqs == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const DecodeKernelInfo* k = pick_decode8(shape, kv_format);
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return PA_ERR_CUDA;
    const size_t need = counters_bytes(shape) + partials_bytes(shape, ctas);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;
    // every (block, head) piece is bulk-copied from p.kv8; the tensor-map
    // parameters of the kernel go unused
    CUtensorMap unused{};

    DecodeLaunch L{};
    L.tmap_k = &unused;
    L.tmap_v = &unused;
    L.p.q = static_cast<const uint16_t*>(q);
    L.p.block_tables = block_tables;
    L.p.context_lens = context_lens;
    L.p.out = static_cast<uint16_t*>(out);
    L.p.counters = static_cast<int32_t*>(workspace);
    L.p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counters_bytes(shape));
    L.p.err = err_word;
    L.p.kv8 = static_cast<const uint8_t*>(kv_pool);
    L.p.v_scale = v_scale;
    L.p.N = shape->num_seqs;
    L.p.Hq = shape->num_q_heads;
    L.p.Hkv = shape->num_kv_heads;
    L.p.NB = shape->num_blocks;
    L.p.MB = shape->max_blocks_per_seq;
    // K's scale folds into the scores: s = scale * k_scale * <q, code>
    L.p.scale_log2 = (float)((double)scale * (double)k_scale * 1.4426950408889634);
    L.p.timeout_ns = kTimeoutNs;
    L.stream = static_cast<cudaStream_t>(stream);
    L.grid = ctas;
    if (cudaMemsetAsync(workspace, 0, counters_bytes(shape), L.stream) != cudaSuccess) return PA_ERR_CUDA;
    return k->launch(L) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_append_kv_fp8(const pa_shape* shape, int32_t kv_format, int32_t num_tokens, const void* k_new,
                           const void* v_new, const int64_t* slot_mapping, void* kv_pool, float k_scale,
                           float v_scale, uint32_t* err_word, void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if (elem_bytes(shape->dtype) != 2 || num_tokens < 0) return PA_ERR_INVALID_ARG;
    st = check_fp8(shape, kv_format, k_scale, v_scale);
    if (st != PA_OK) return st;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_pool) return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_pool, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    Append8Args a;
    a.T = num_tokens;
    a.Hkv = shape->num_kv_heads;
    a.D = shape->head_dim;
    a.BS = shape->block_size;
    a.num_slots = (long long)shape->num_blocks * shape->block_size;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.err = err_word;
    return append8_launch(k_new, v_new, slot_mapping, kv_pool, a, shape->dtype == PA_BF16,
                          kv_format == PA_FP8_E5M2, static_cast<cudaStream_t>(stream), sms) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_append_kv(const pa_shape* shape, int32_t num_tokens, const void* k_new, const void* v_new,
                       const int64_t* slot_mapping, void* k_pool, void* v_pool, uint32_t* err_word,
                       void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if (elem_bytes(shape->dtype) != 2 || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    AppendArgs a;
    a.T = num_tokens;
    a.Hkv = shape->num_kv_heads;
    a.vec_per_row = shape->head_dim * 2 / 16;
    a.BS = shape->block_size;
    a.num_slots = (long long)shape->num_blocks * shape->block_size;
    a.err = err_word;
    return append_launch(k_new, v_new, slot_mapping, k_pool, v_pool, a, static_cast<cudaStream_t>(stream), sms) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_copy_blocks_fp8(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs,
                             void* kv_pool, uint32_t* err_word, void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if ((shape->dtype != PA_FP8_E4M3 && shape->dtype != PA_FP8_E5M2) || num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!src_dst_pairs || !kv_pool || !aligned(kv_pool, 16) || !aligned(src_dst_pairs, 4)) return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    CopyArgs a;
    a.n = num_pairs;
    a.vec_per_block = (long long)shape->num_kv_heads * 2 * shape->block_size * shape->head_dim / 16;   // bytes / 16
    a.NB = shape->num_blocks;
    a.err = err_word;
    return copy_launch(src_dst_pairs, kv_pool, nullptr, a, static_cast<cudaStream_t>(stream), sms) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs, void* k_pool,
                         void* v_pool, uint32_t* err_word, void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if (elem_bytes(shape->dtype) != 2 || num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!src_dst_pairs || !k_pool || !v_pool) return PA_ERR_INVALID_ARG;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(src_dst_pairs, 4)) return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    CopyArgs a;
    a.n = num_pairs;
    a.vec_per_block = (long long)shape->num_kv_heads * shape->block_size * shape->head_dim * 2 / 16;
    a.NB = shape->num_blocks;
    a.err = err_word;
    return copy_launch(src_dst_pairs, k_pool, v_pool, a, static_cast<cudaStream_t>(stream), sms) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_read_error(const uint32_t* err_word, void* stream) {
    if (!err_word) return PA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, err_word, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
    if (w & PA_DEVERR_TIMEOUT) return PA_ERR_TIMEOUT;
    if (w) return PA_ERR_OUT_OF_RANGE;
    return PA_OK;
}

const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_OUT_OF_RANGE: return "out-of-range data found on the device";
        case PA_ERR_TIMEOUT: return "device wait timed out";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int32_t pa_version(void) { return 100; }

}  // extern "C"
