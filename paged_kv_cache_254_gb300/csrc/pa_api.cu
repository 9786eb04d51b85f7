// C ABI of libpa (declared in include/pa.h): host-side argument checks,
// kernel selection, TMA descriptor set-up and launches.  Nothing here
// allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/pa.h"
#include "decode_kernel.cuh"
#include "kv_ops.cuh"
#include "multi_kernel.cuh"
#include "multi_tc_kernel.cuh"
#include "prefix_kernel.cuh"

namespace {

using namespace pa;

constexpr uint64_t kTimeoutNs = 2000000000ull;   // bound on any device-side wait
constexpr uint64_t kMaxStallNs = 1000000000ull;  // longest injected stall (pa_set_decode_stall_ns)

// Injected stall of the decode kernel's first stage wait (0: off).
std::atomic<uint64_t> g_stall_ns{0};

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

// ---------------------------------------------------------------- decode scratch
// One region per decode launch: the dynamic-chunk counter, per-sequence block
// prefix sums, and two partial states (o[d], m, l per query row of a group,
// rows of d + 4 floats) per chunk.  Chunks: one per worker warp, plus up to
// kDynPerWorker per worker claimed at run time.
constexpr int kDynPerWorker = 4;

size_t counters_bytes(const pa_shape*) { return 256; }

size_t cum_bytes(const pa_shape* s) {
    const size_t c = ((size_t)s->num_seqs + 1) * sizeof(long long);
    return (c + 255) & ~size_t(255);
}

size_t piece_bytes(const pa_shape* s) {
    const int g = s->num_q_heads / s->num_kv_heads;
    return (size_t)2 * g * (s->head_dim + 4) * sizeof(float);
}

// Region size for `workers` static chunks and `nd` dynamic ones.
size_t decode_region_bytes(const pa_shape* s, long long workers, long long nd) {
    return counters_bytes(s) + cum_bytes(s) + (size_t)(workers + nd) * piece_bytes(s);
}

// Zero the chunk counter; cum[s] = blocks of the
// sequences before s in the decode work list (with a shared-prefix pass,
// blocks after each sequence's first_blocks).  One CTA.
__global__ void __launch_bounds__(1024)
pa_decode_prepass(const int32_t* __restrict__ context_lens, const int32_t* __restrict__ first_blocks, int N,
                  int MB, int BS, int32_t* __restrict__ counters, long long n_counters,
                  long long* __restrict__ cum) {
    __shared__ long long wsum[32];
    __shared__ long long carry;
    griddep_launch_dependents();   // the attention kernel may set up meanwhile; it waits for this grid
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (long long i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
    if (threadIdx.x == 0) {
        carry = 0;
        cum[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int s = base + (int)threadIdx.x;
        long long v = 0;
        if (s < N) {
            const int c = context_lens[s];
            const int nb = (c > 0 && c <= MB * BS) ? (c + BS - 1) / BS : 0;
            const int f = first_blocks ? first_blocks[s] : 0;
            v = nb - f > 0 ? nb - f : 0;
        }
        long long x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += t;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            long long w = wsum[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const long long t = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += t;
            }
            wsum[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const long long incl = carry + (warp > 0 ? wsum[warp - 1] : 0) + x;
        if (s < N) cum[s + 1] = incl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
}

template <int D>
cudaError_t merge_launch(const DecodeLaunch& L, int g, long long nworkers, cudaStream_t st) {
    constexpr int HPW = 32 / (D / 4);
    const long long tasks = (long long)L.p.N * L.p.Hkv * ((g + HPW - 1) / HPW);
    const long long blocks = (tasks + 7) / 8;
    // programmatic stream serialization: the merge's CTAs are placed as the
    // decode's retire, then wait for the decode grid (griddep_wait)
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(blocks, 256, 0, st, attr);
    return cudaLaunchKernelEx(&cfg, pa_decode_merge<D>, L.p.cum, static_cast<const float*>(L.p.partials), L.p.out,
                              L.p.N, L.p.Hkv, g, nworkers, L.p.nd, L.p.v_scale, L.bf16 ? 1 : 0);
}

// Lay out the decode region, run the pre-pass, fill L's scheduling fields,
// launch the decode and the merge of split pairs.  L's other fields are set
// by the caller.
pa_status run_decode(const DecodeKernelInfo* k, int ctas, DecodeLaunch& L, const pa_shape* s, void* region,
                     size_t region_bytes, const int32_t* first_blocks) {
    const long long workers = (long long)ctas * k->workers;
    const size_t fixed = counters_bytes(s) + cum_bytes(s);
    if (!region || region_bytes < decode_region_bytes(s, workers, 0)) return PA_ERR_WORKSPACE;
    long long cap = (long long)((region_bytes - fixed) / piece_bytes(s)) - workers;
    long long nd = kDynPerWorker * workers;
    if (nd > cap) nd = cap;
    if (nd > (1ll << 30)) nd = 1ll << 30;
    uint8_t* base = static_cast<uint8_t*>(region);
    L.p.chunk_ctr = reinterpret_cast<int32_t*>(base);
    L.p.cum = reinterpret_cast<const long long*>(base + counters_bytes(s));
    L.p.partials = reinterpret_cast<float*>(base + fixed);
    L.p.nd = (int32_t)nd;
    L.p.stall_ns = g_stall_ns.load(std::memory_order_relaxed);
    L.grid = ctas;
    L.bf16 = s->dtype == PA_BF16;
    pa_decode_prepass<<<1, 1024, 0, L.stream>>>(L.p.context_lens, first_blocks, s->num_seqs,
                                                s->max_blocks_per_seq, s->block_size, L.p.chunk_ctr, 1,
                                                const_cast<long long*>(L.p.cum));
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (k->launch(L) != cudaSuccess) return PA_ERR_CUDA;
    const int g = s->num_q_heads / s->num_kv_heads;
    const cudaError_t e = s->head_dim == 128 ? merge_launch<128>(L, g, workers, L.stream)
                                             : merge_launch<64>(L, g, workers, L.stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
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

// The pool as a 3-D tensor (column within a 64-column half, row = (block,
// kv head, slot), half): one box of 64 columns x block_size rows x all halves
// lands as the halves' 128-byte swizzled [rows][128 B] tiles one after the
// other -- a whole (block, kv head) chunk in one copy.  The half stride
// (128 bytes) is below the row stride.
bool pool_map_chunk(CUtensorMap* m, const void* pool, const pa_shape* s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int halves = s->head_dim / 64;
    const cuuint64_t dims[3] = {64, (cuuint64_t)s->num_blocks * s->num_kv_heads * s->block_size, (cuuint64_t)halves};
    const cuuint64_t strides[2] = {(cuuint64_t)s->head_dim * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)s->block_size, (cuuint32_t)halves};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The pool as a 4-D tensor (column within a 64-column half, row within an
// 8-row group, half, 8-row group): one box of 64 columns x 8 rows x all halves
// x block_size / 8 groups lands a whole (block, kv head) chunk as
// [group][half][8 rows][128 B], one 1024-byte swizzle atom per (group, half).
// Consecutive 8-row groups of a half are then a fixed stride apart (halves x
// 1024 bytes) across the blocks of a stage, so one K-major descriptor spans
// all of a stage's keys.
bool pool_map_groups(CUtensorMap* m, const void* pool, const pa_shape* s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int halves = s->head_dim / 64;
    const cuuint64_t rows = (cuuint64_t)s->num_blocks * s->num_kv_heads * s->block_size;
    const cuuint64_t dims[4] = {64, 8, (cuuint64_t)halves, rows / 8};
    const cuuint64_t strides[3] = {(cuuint64_t)s->head_dim * 2, 128, (cuuint64_t)s->head_dim * 2 * 8};
    const cuuint32_t box[4] = {64, 8, (cuuint32_t)halves, (cuuint32_t)s->block_size / 8};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 4, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [T][Hq][D] as a 3-D tensor (head_dim, heads, tokens): boxes of 64
// columns x g heads x q_box tokens land as rows i * g + hh, 128-byte swizzled.
bool q_map(CUtensorMap* m, const void* q, const pa_shape* s, int total_q, int q_box) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int g = s->num_q_heads / s->num_kv_heads;
    const cuuint64_t dims[3] = {(cuuint64_t)s->head_dim, (cuuint64_t)s->num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {(cuuint64_t)s->head_dim * 2, (cuuint64_t)s->num_q_heads * s->head_dim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)q_box};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
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

// 4-bit cache: queries and new values in the shape's 16-bit dtype, head_dim 128.
pa_status check_int4(const pa_shape* s) {
    if (s->dtype != PA_FP16 && s->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (s->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (s->block_size != 16 && s->block_size != 32) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

int int4_piece_bytes(const pa_shape* s) { return s->block_size * s->head_dim + 8 * s->block_size; }

const DecodeKernelInfo* pick_decode4(const pa_shape* s) {
    static const auto tab = [] {
        struct T { DecodeKernelInfo bf[2][5], fp[2][5]; } x;
        decode4_table_bf16(x.bf);
        decode4_table_fp16(x.fp);
        return x;
    }();
    const int lg = log2_exact(s->num_q_heads / s->num_kv_heads);
    const int b = s->block_size == 32 ? 1 : 0;
    return s->dtype == PA_BF16 ? &tab.bf[b][lg] : &tab.fp[b][lg];
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

// ---------------------------------------------------------------- multi-token query
// Launches whose (sequence, KV head) pairs carry more than 16 query rows
// (max_q * g) run on the tensor-core (tcgen05) kernel: 128-row MMA tiles, one
// CTA per SM.  Up to 16 rows, the mma.sync kernel's single 16-row tile per
// pair reads each block once for all rows and stays close to the HBM bound;
// above that its tiles double the MMA and softmax work per block while the
// tcgen05 tile costs the same up to 128 rows (70B-shaped batch, 4-token
// chunks: 1.09 ms on two mma.sync tiles, 0.86 ms on tcgen05).
constexpr int kTcMinRows = 17;

// Shape rules shared by both multi-token kernels; `rows` = max_q * g.
pa_status check_multi(const pa_shape* s, int max_q, int* rows) {
    const DecodeKernelInfo* k16 = nullptr;
    pa_status st = pick_decode(s, &k16);                  // the same shape rules as decode
    if (st != PA_OK) return st;
    if (max_q < 1 || max_q > 16) return PA_ERR_INVALID_ARG;
    *rows = max_q * (s->num_q_heads / s->num_kv_heads);
    return *rows > 128 ? PA_ERR_UNSUPPORTED : PA_OK;
}

// The mma.sync kernel: one 16-row tile per (sequence, KV head) pair.
const MultiKernelInfo* pick_multi(const pa_shape* s) {
    static const auto tab = [] {
        struct T { MultiKernelInfo t[2][2][2]; } x;      // [bf16][d == 128][bs == 32]
        multi_table_fp16_d64(x.t[0][0]);
        multi_table_fp16_d128(x.t[0][1]);
        multi_table_bf16_d64(x.t[1][0]);
        multi_table_bf16_d128(x.t[1][1]);
        return x;
    }();
    return &tab.t[s->dtype == PA_BF16][s->head_dim == 128][s->block_size == 32];
}

const MultiKernelInfo* pick_multi_tc(const pa_shape* s) {
    static const auto tab = [] {
        struct T { MultiKernelInfo t[2][2][2]; } x;      // [bf16][d == 128][bs == 32]
        multi_tc_table_fp16_d64(x.t[0][0]);
        multi_tc_table_fp16_d128(x.t[0][1]);
        multi_tc_table_bf16_d64(x.t[1][0]);
        multi_tc_table_bf16_d128(x.t[1][1]);
        return x;
    }();
    return &tab.t[s->dtype == PA_BF16][s->head_dim == 128][s->block_size == 32];
}

// Scratch of a multi-token launch: chunk counter, block prefix sums, two
// partial states per tile row per CTA.
size_t multi_region_bytes(const pa_shape* s, int ctas, int rows) {
    return counters_bytes(s) + cum_bytes(s) + (size_t)ctas * 2 * rows * (s->head_dim + 4) * sizeof(float);
}

// Workspace of prefix-aware decode (offsets in off[]): [0] prefix counters,
// [1] first block per sequence (both zeroed before the prefix pass), [2] carry
// states, [3] prefix partials, [4] the decode region (to the end).
size_t shared_prefix_layout(const pa_shape* s, long long dec_workers, int pre_ctas, size_t (&off)[5]) {
    off[0] = 0;
    off[1] = align256((size_t)s->num_seqs * s->num_kv_heads * sizeof(int32_t));
    off[2] = off[1] + align256((size_t)s->num_seqs * sizeof(int32_t));
    const size_t carry = align256((size_t)s->num_seqs * s->num_q_heads * (s->head_dim + 2) * sizeof(float));
    off[3] = off[2] + carry;
    off[4] = off[3] + align256((size_t)pre_ctas * 2 * 32 * (s->head_dim + 2) * sizeof(float));
    return off[4] + decode_region_bytes(s, dec_workers, kDynPerWorker * dec_workers);
}

}  // namespace

namespace pa {

// Smallest scratch pa_decode accepts for `shape` on the current device (one
// chunk per worker warp), or 0 with *why set when the shape is invalid or
// unsupported (its status) or a CUDA query fails (PA_ERR_CUDA).
size_t decode_min_workspace_bytes(const pa_shape* shape, pa_status* why) {
    const DecodeKernelInfo* k = nullptr;
    const pa_status st = pick_decode(shape, &k);
    if (st != PA_OK) {
        *why = st;
        return 0;
    }
    int dev = 0;
    const int ctas = cudaGetDevice(&dev) == cudaSuccess ? k->max_ctas(dev) : -1;
    if (ctas <= 0) {
        *why = PA_ERR_CUDA;
        return 0;
    }
    *why = PA_OK;
    return decode_region_bytes(shape, (long long)ctas * k->workers, 0);
}

}  // namespace pa

extern "C" {

pa_status pa_set_decode_stall_ns(uint64_t wait_ns) {
    if (wait_ns > kMaxStallNs) return PA_ERR_INVALID_ARG;
    g_stall_ns.store(wait_ns, std::memory_order_relaxed);
    return PA_OK;
}

size_t pa_decode_workspace_bytes(const pa_shape* shape) {
    const DecodeKernelInfo* k = nullptr;
    if (pick_decode(shape, &k) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return 0;
    const long long workers = (long long)ctas * k->workers;
    return decode_region_bytes(shape, workers, kDynPerWorker * workers);
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
    if (!workspace || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!pool_map_chunk(&mk, k_pool, shape) || !pool_map_chunk(&mv, v_pool, shape)) return PA_ERR_CUDA;

    DecodeLaunch L{};
    L.tmap_k = &mk;
    L.tmap_v = &mv;
    L.p.q = static_cast<const uint16_t*>(q);
    L.p.block_tables = block_tables;
    L.p.context_lens = context_lens;
    L.p.out = static_cast<uint16_t*>(out);
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
    // The counters start at zero for every call (the pre-pass clears them;
    // the region may hold another shape's state from an earlier call).
    return run_decode(k, ctas, L, shape, workspace, workspace_bytes, nullptr);
}

size_t pa_decode_shared_prefix_workspace_bytes(const pa_shape* shape) {
    const DecodeKernelInfo* k = nullptr;
    if (pick_decode(shape, &k) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int dec = k->max_ctas(dev), pre = pick_prefix(shape).max_ctas(dev);
    if (dec <= 0 || pre <= 0) return 0;
    size_t off[5];
    return shared_prefix_layout(shape, (long long)dec * k->workers, pre, off);
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
    size_t off[5];
    shared_prefix_layout(shape, (long long)dec * k->workers, pre, off);
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < off[4] + decode_region_bytes(shape, (long long)dec * k->workers, 0))
        return PA_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!pool_map_chunk(&mk, k_pool, shape) || !pool_map_chunk(&mv, v_pool, shape)) return PA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    const float scale_log2 = (float)((double)scale * 1.4426950408889634);   // log2(e)
    // the prefix arrival counters and the first-block array start at zero
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
        P.p.first_blocks = reinterpret_cast<int32_t*>(ws + off[1]);
        P.p.counters = reinterpret_cast<int32_t*>(ws + off[0]);
        P.p.partials = reinterpret_cast<float*>(ws + off[3]);
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
    L.p.err = err_word;
    L.p.first_blocks = reinterpret_cast<const int32_t*>(ws + off[1]);
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
    return run_decode(k, dec, L, shape, ws + off[4], workspace_bytes - off[4], L.p.first_blocks);
}

size_t pa_decode_fp8_workspace_bytes(const pa_shape* shape, int32_t kv_format) {
    const DecodeKernelInfo* k16 = nullptr;
    if (pick_decode(shape, &k16) != PA_OK || check_fp8(shape, kv_format, 1.f, 1.f) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const DecodeKernelInfo* k8 = pick_decode8(shape, kv_format);
    const int ctas = k8->max_ctas(dev);
    if (ctas <= 0) return 0;
    const long long workers = (long long)ctas * k8->workers;
    return decode_region_bytes(shape, workers, kDynPerWorker * workers);
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
    if (!workspace || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
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
    return run_decode(k, ctas, L, shape, workspace, workspace_bytes, nullptr);
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


size_t pa_decode_multi_workspace_bytes(const pa_shape* shape, int32_t max_q_len) {
    int rows = 0;
    if (check_multi(shape, max_q_len, &rows) != PA_OK) return 0;
    const MultiKernelInfo* k = pick_multi(shape);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return 0;
    size_t need = multi_region_bytes(shape, ctas, k->rows);
    if (rows >= kTcMinRows) {
        const MultiKernelInfo* t = pick_multi_tc(shape);
        const int tctas = t->max_ctas(dev);
        if (tctas <= 0) return 0;
        need = std::max(need, multi_region_bytes(shape, tctas, t->rows));
    }
    return need;
}

pa_status pa_decode_multi(const pa_shape* shape, int32_t max_q_len, int32_t total_q, const void* q,
                          const int32_t* q_start, const void* k_pool, const void* v_pool,
                          const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                          void* workspace, size_t workspace_bytes, uint32_t* err_word, void* stream) {
    int g_rows = 0;
    pa_status st = check_multi(shape, max_q_len, &g_rows);
    if (st != PA_OK) return st;
    if (total_q < 0) return PA_ERR_INVALID_ARG;
    // with no query rows at all (total_q 0) the mma.sync kernel only checks
    // the chunk descriptions: every chunk is empty or malformed
    const bool tc = g_rows >= kTcMinRows && total_q > 0;
    const MultiKernelInfo* k = tc ? pick_multi_tc(shape) : pick_multi(shape);
    if (!q_start || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (total_q > 0 && (!q || !out)) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(q_start, 4))
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->num_seqs == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return PA_ERR_CUDA;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < multi_region_bytes(shape, ctas, k->rows))
        return PA_ERR_WORKSPACE;
    CUtensorMap mk, mv, mq;
    // the tcgen05 kernel copies K and V as whole (block, kv head) chunks: K in
    // 8-row groups (one descriptor spans a stage's keys), V as column halves
    if (!(tc ? pool_map_groups(&mk, k_pool, shape) : pool_map_chunk(&mk, k_pool, shape)) ||
        !pool_map_chunk(&mv, v_pool, shape))
        return PA_ERR_CUDA;
    const int q_box = std::min(max_q_len, total_q);
    if (tc && !q_map(&mq, q, shape, total_q, q_box)) return PA_ERR_CUDA;

    uint8_t* base = static_cast<uint8_t*>(workspace);
    MultiLaunch L{};
    L.tmap_q = tc ? &mq : nullptr;
    L.tmap_k = &mk;
    L.tmap_v = &mv;
    DecodeParams& d = L.p.d;
    d.q = static_cast<const uint16_t*>(q);
    d.block_tables = block_tables;
    d.context_lens = context_lens;
    d.out = static_cast<uint16_t*>(out);
    d.err = err_word;
    d.chunk_ctr = reinterpret_cast<int32_t*>(base);
    d.cum = reinterpret_cast<const long long*>(base + counters_bytes(shape));
    d.partials = reinterpret_cast<float*>(base + counters_bytes(shape) + cum_bytes(shape));
    d.N = shape->num_seqs;
    d.Hq = shape->num_q_heads;
    d.Hkv = shape->num_kv_heads;
    d.NB = shape->num_blocks;
    d.MB = shape->max_blocks_per_seq;
    d.scale_log2 = (float)((double)scale * 1.4426950408889634);   // log2(e)
    d.timeout_ns = kTimeoutNs;
    d.v_scale = 1.0f;
    L.p.q_start = q_start;
    L.p.max_q = max_q_len;
    L.p.total_q = total_q;
    L.p.q_box = q_box;
    L.stream = static_cast<cudaStream_t>(stream);
    L.grid = ctas;
    pa_decode_prepass<<<1, 1024, 0, L.stream>>>(context_lens, nullptr, shape->num_seqs,
                                                shape->max_blocks_per_seq, shape->block_size, d.chunk_ctr, 1,
                                                const_cast<long long*>(d.cum));
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (k->launch(L) != cudaSuccess) return PA_ERR_CUDA;
    const int g = shape->num_q_heads / shape->num_kv_heads;
    if (ctas > 1) {   // one CTA per chunk boundary: the pairs cut there
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = pdl_config(ctas - 1, MERGE_THREADS, 0, L.stream, attr);
        const float* parts = d.partials;
        const int bf = shape->dtype == PA_BF16;
        const cudaError_t e =
            shape->head_dim == 128
                ? cudaLaunchKernelEx(&cfg, pa_multi_merge<128>, d.cum, q_start, context_lens, parts, d.out, d.N,
                                     d.Hkv, g, k->rows, ctas, max_q_len, total_q, bf)
                : cudaLaunchKernelEx(&cfg, pa_multi_merge<64>, d.cum, q_start, context_lens, parts, d.out, d.N, d.Hkv,
                                     g, k->rows, ctas, max_q_len, total_q, bf);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}


size_t pa_decode_int4_workspace_bytes(const pa_shape* shape) {
    const DecodeKernelInfo* k16 = nullptr;
    if (pick_decode(shape, &k16) != PA_OK || check_int4(shape) != PA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const DecodeKernelInfo* k4 = pick_decode4(shape);
    const int ctas = k4->max_ctas(dev);
    if (ctas <= 0) return 0;
    const long long workers = (long long)ctas * k4->workers;
    return decode_region_bytes(shape, workers, kDynPerWorker * workers);
}

pa_status pa_decode_int4(const pa_shape* shape, const void* q, const void* kv_pool, const int32_t* block_tables,
                         const int32_t* context_lens, float scale, void* out, void* workspace,
                         size_t workspace_bytes, uint32_t* err_word, void* stream) {
    const DecodeKernelInfo* k16 = nullptr;
    pa_status st = pick_decode(shape, &k16);
    if (st != PA_OK) return st;
    st = check_int4(shape);
    if (st != PA_OK) return st;
    if (!q || !kv_pool || !block_tables || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->num_seqs == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const DecodeKernelInfo* k = pick_decode4(shape);
    const int ctas = k->max_ctas(dev);
    if (ctas <= 0) return PA_ERR_CUDA;
    if (!workspace || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    CUtensorMap unused{};   // every (block, head) piece is bulk-copied from p.kv8
    DecodeLaunch L{};
    L.tmap_k = &unused;
    L.tmap_v = &unused;
    L.p.q = static_cast<const uint16_t*>(q);
    L.p.block_tables = block_tables;
    L.p.context_lens = context_lens;
    L.p.out = static_cast<uint16_t*>(out);
    L.p.err = err_word;
    L.p.kv8 = static_cast<const uint8_t*>(kv_pool);
    L.p.v_scale = 1.0f;                              // per-row scales are applied inside
    L.p.N = shape->num_seqs;
    L.p.Hq = shape->num_q_heads;
    L.p.Hkv = shape->num_kv_heads;
    L.p.NB = shape->num_blocks;
    L.p.MB = shape->max_blocks_per_seq;
    L.p.scale_log2 = (float)((double)scale * 1.4426950408889634);   // log2(e)
    L.p.timeout_ns = kTimeoutNs;
    L.stream = static_cast<cudaStream_t>(stream);
    return run_decode(k, ctas, L, shape, workspace, workspace_bytes, nullptr);
}

pa_status pa_append_kv_int4(const pa_shape* shape, int32_t num_tokens, const void* k_new, const void* v_new,
                            const int64_t* slot_mapping, void* kv_pool, uint32_t* err_word, void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    st = check_int4(shape);
    if (st != PA_OK) return st;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_pool) return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_pool, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    Append4Args a;
    a.T = num_tokens;
    a.Hkv = shape->num_kv_heads;
    a.BS = shape->block_size;
    a.piece_bytes = int4_piece_bytes(shape);
    a.num_slots = (long long)shape->num_blocks * shape->block_size;
    a.err = err_word;
    return append4_launch(k_new, v_new, slot_mapping, kv_pool, a, shape->dtype == PA_BF16,
                          static_cast<cudaStream_t>(stream), sms) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_copy_blocks_int4(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs,
                              void* kv_pool, uint32_t* err_word, void* stream) {
    pa_status st = check_common(shape);
    if (st != PA_OK) return st;
    if (num_pairs < 0) return PA_ERR_INVALID_ARG;
    st = check_int4(shape);
    if (st != PA_OK) return st;
    if (num_pairs == 0) return PA_OK;
    if (!src_dst_pairs || !kv_pool || !aligned(kv_pool, 16) || !aligned(src_dst_pairs, 4)) return PA_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    CopyArgs a;
    a.n = num_pairs;
    a.vec_per_block = (long long)shape->num_kv_heads * int4_piece_bytes(shape) / 16;   // bytes / 16
    a.NB = shape->num_blocks;
    a.err = err_word;
    return copy_launch(src_dst_pairs, kv_pool, nullptr, a, static_cast<cudaStream_t>(stream), sms) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

}  // extern "C"
