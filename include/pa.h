/*
 * pa.h -- C ABI of libpa: paged KV-cache decode attention for sm_103a (GB300).
 *
 * The KV cache is a pool of fixed-size physical blocks; a sequence reaches its
 * tokens through a block table (logical block i = floor(t / B), offset
 * j = t mod B).  Sources: "vLLM & High-Throughput Serving ..." (thewebvale.com),
 * section 2 "PagedAttention: Virtual Memory Virtualization ...", block-table
 * formula; "AI Inference Serving at Scale ..." (ontq.xyz), section 3
 * "PagedAttention: Virtual Memory and Paging for GPU Tensors".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor argument is a DEVICE pointer to contiguous row-major memory
 *    owned by the caller.  The library allocates nothing and keeps no
 *    per-call state between calls (it caches per-device launch properties).
 *  - 16-bit element pointers (q, pools, out, new K/V) must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work on `stream` and return; the caller synchronises.
 *  - Host-side argument checks run before any launch; a failing check returns
 *    its status and enqueues nothing.
 *  - Bad data found on the device (a block id outside [0, num_blocks), a
 *    context length outside [0, max_blocks_per_seq * block_size], a slot past
 *    the pool, a bad copy pair) never traps: the kernel ORs a PA_DEVERR_* bit
 *    into `*err_word` (if err_word is not NULL), skips the bad access, and
 *    writes NaN to the affected decode rows.  pa_read_error() turns the word
 *    into a status.
 *
 * Pool layout: k_pool and v_pool are [num_blocks][num_kv_heads][block_size]
 * [head_dim]; one (block, kv head) chunk is block_size * head_dim contiguous
 * elements.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, misaligned pointer, Hq % Hkv != 0 */
    PA_ERR_UNSUPPORTED = 2,   /* a shape outside the compiled set (see pa_decode) */
    PA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    PA_ERR_OUT_OF_RANGE = 4,  /* device found a bad block id, context length, slot or copy pair */
    PA_ERR_TIMEOUT = 5,       /* a device-side wait ran past its limit; the kernel gave up */
    PA_ERR_WORKSPACE = 6      /* workspace missing, misaligned or below the shape's minimum */
} pa_status;

/* Element types.  PA_FP16 / PA_BF16: queries, outputs, new keys and values,
 * and the 16-bit cache.  PA_FP8_E4M3 / PA_FP8_E5M2: the 8-bit cache formats
 * (kv_format arguments of the *_fp8 entry points). */
typedef enum pa_dtype { PA_FP16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2, PA_FP8_E5M2 = 3 } pa_dtype;

/* Bits ORed into *err_word by the kernels. */
#define PA_DEVERR_BLOCK_ID  1u   /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT   2u   /* context length < 0 or > max_blocks_per_seq * block_size */
#define PA_DEVERR_SLOT      4u   /* slot >= num_blocks * block_size */
#define PA_DEVERR_COPY_PAIR 8u   /* copy pair id outside [0, num_blocks) */
#define PA_DEVERR_TIMEOUT   16u  /* a bounded wait expired */
#define PA_DEVERR_GROUP     32u  /* prefix group malformed, or a member does not share the prefix */
#define PA_DEVERR_Q_RANGE   64u  /* a bf16 query element beyond fp16's finite range (8-bit and 4-bit
                                    caches, which compute in fp16); its rows are not finite */

typedef struct pa_shape {
    int32_t num_seqs;            /* N: sequences in the batch (>= 0) */
    int32_t num_q_heads;         /* Hq */
    int32_t num_kv_heads;        /* Hkv; query head h reads KV head h / (Hq / Hkv) */
    int32_t head_dim;            /* d */
    int32_t block_size;          /* B: tokens per physical block */
    int32_t num_blocks;          /* NB: blocks in the pool */
    int32_t max_blocks_per_seq;  /* MB: columns of the block table */
    int32_t dtype;               /* pa_dtype of q, pools, out and new K/V */
} pa_shape;

/*
 * Bytes of scratch that pa_decode prefers for `shape` on the CURRENT device.
 * The workspace holds a work-chunk counter, the per-sequence block prefix
 * sums that place the work chunks, and the partial
 * softmax states of sequences whose keys are split across chunks.  It needs
 * no initialisation: pa_decode's first launch (a one-block pre-pass on
 * `stream`) clears the counter and writes the prefix sums; the attention
 * kernel follows, then a merge kernel for the sequences split across chunks
 * (three launches on `stream` in all).  A smaller
 * workspace is accepted down to the static split's minimum (one chunk per
 * worker warp); below the preferred size fewer chunks are balanced at run
 * time, and results are deterministic for each workspace size.  The same
 * buffer can serve any later call on the same stream, whatever its shape;
 * calls that may run at the same time must use different workspaces.  Returns
 * 0 if the shape is invalid or unsupported.
 */
size_t pa_decode_workspace_bytes(const pa_shape* shape);

/*
 * Paged decode attention ("How LLM Inference Engines Work ..." by
 * letsbuildsolutions.com, section "PagedAttention: Virtual Memory for KV
 * Caches": the kernel gathers K and V from non-adjacent blocks; ontq section 8:
 * the result equals un-paged attention; ontq section 6: grouped-query heads).
 *
 * For each sequence b and query head h, with g = Hq / Hkv, kh = h / g and
 * n = context_lens[b]:
 *     s_t  = scale * <q[b,h,:], K_pool[table[b][t/B], kh, t%B, :]>,  t < n
 *     out[b,h,:] = sum_t softmax(s)_t * V_pool[table[b][t/B], kh, t%B, :]
 * accumulated in fp32 and rounded once to the output dtype.  n == 0 gives a
 * zero row.  Table entries past ceil(n / B) and pool slots past position n-1
 * are never read.
 *
 *   q             [N][Hq][d]            query of the newest token
 *   k_pool,v_pool [NB][Hkv][B][d]       the cache
 *   block_tables  int32 [N][MB]         physical block ids in logical order
 *   context_lens  int32 [N]             tokens cached per sequence (incl. the newest)
 *   scale         fp32 softmax scale (typically 1/sqrt(d))
 *   out           [N][Hq][d]            result, same dtype as q
 *   workspace     see pa_decode_workspace_bytes
 *   err_word      device uint32, may be NULL
 *
 * Supported: dtype fp16 or bf16; d in {64, 128}; B in {16, 32};
 * g in {1, 2, 4, 8, 16}; NB * Hkv * B < 2^31.  Others: PA_ERR_UNSUPPORTED.
 * Results are deterministic for a given device and input, and bitwise
 * independent of where the blocks sit in the pool.
 */
pa_status pa_decode(const pa_shape* shape, const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    void* out, void* workspace, size_t workspace_bytes, uint32_t* err_word,
                    void* stream);

/*
 * 4-bit integer (INT4) KV cache.  Compressing keys and values to 4 bits
 * quadruples the requests that fit (ontq "AI Inference Serving at Scale",
 * section 6); 4-bit integer formats carry per-group scale factors
 * (letsbuildsolutions "How LLM Inference Engines Work", quantization).
 * Format: one group per cached (token, KV head) row of K or of V, scale =
 * amax / 7 (fp32), code = nearest integer to x / scale (fp32 division, ties to
 * even) in [-8, 7]; a zero row has scale 0.  Decoding: code * scale.
 * Layout: ONE pool of bytes [NB][Hkv][P] with P = B * d + 8 * B; each
 * (block, KV head) piece holds the K codes token-major (B rows of d / 2
 * bytes), the V codes dims-first (d rows of B / 2 bytes), then B fp32 K
 * scales and B fp32 V scales.  Codes are stored as nibbles code + 8; in each
 * little-endian 32-bit word of 8 elements, element 2k is nibble k and element
 * 2k + 1 is nibble k + 4.  Supported: head_dim 128, B in {16, 32}, g in
 * {1, 2, 4, 8, 16}; shape->dtype is the 16-bit type of q, out and new K/V.
 *
 * pa_append_kv_int4: quantize k_new / v_new ([T][Hkv][d]) into the pool at
 * slot_mapping (negative skips; past the pool: PA_DEVERR_SLOT).
 * pa_decode_int4: pa_decode over the 4-bit pool (attention over the decoded
 * values); fp16 tensor-core arithmetic on the codes (q rounded to fp16; a bf16
 * query beyond fp16's finite range sets PA_DEVERR_Q_RANGE), the K scale
 * applied to each score and the V scale to each softmax weight, fp32
 * accumulation.
 * pa_copy_blocks_int4: copy-on-write copies of whole blocks of the pool.
 */
size_t pa_decode_int4_workspace_bytes(const pa_shape* shape);

pa_status pa_decode_int4(const pa_shape* shape, const void* q, const void* kv_pool,
                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                         void* out, void* workspace, size_t workspace_bytes, uint32_t* err_word,
                         void* stream);

pa_status pa_append_kv_int4(const pa_shape* shape, int32_t num_tokens, const void* k_new,
                            const void* v_new, const int64_t* slot_mapping, void* kv_pool,
                            uint32_t* err_word, void* stream);

pa_status pa_copy_blocks_int4(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs,
                              void* kv_pool, uint32_t* err_word, void* stream);

/*
 * Multi-token query paged attention: a chunk of new tokens per sequence
 * (chunked prefill -- thewebvale "vLLM & High-Throughput Serving", section 4;
 * speculative verification -- letsbuildsolutions "How LLM Inference Engines
 * Work", speculative decoding, where the target model scores every drafted
 * token in one pass).
 *
 * Sequence b brings n_b = q_start[b + 1] - q_start[b] query tokens, its last
 * n_b cached tokens (their K/V appended before the call), at rows
 * q_start[b] .. q_start[b + 1] - 1 of q and out.  Query token i of the chunk
 * attends causally to the keys t <= context_lens[b] - n_b + i:
 *     s_t  = scale * <q[q_start[b] + i, h, :], K(b, t, h / g)>
 *     out[q_start[b] + i, h, :] = sum_t softmax(s)_t * V(b, t, h / g)
 * with K(b, t, kh) = K_pool[table[b][t/B], kh, t%B, :] as in pa_decode.
 *
 *   max_q_len     largest n_b of the call, 1..16; max_q_len * g <= 128
 *   total_q       T: rows of q and out (q_start[N] should equal it)
 *   q, out        [T][Hq][d], same 16-bit dtype as the pools
 *   q_start       device int32 [N + 1], non-decreasing
 *   others        as pa_decode; workspace: pa_decode_multi_workspace_bytes
 *
 * A sequence whose chunk is malformed (n_b < 0, n_b > max_q_len, n_b > its
 * context, rows outside [0, T)) or whose context is invalid sets
 * PA_DEVERR_CONTEXT; its rows inside [0, T) are NaN.  Supported shapes as
 * pa_decode (16-bit); larger max_q_len * g: PA_ERR_UNSUPPORTED.  Three
 * launches on `stream` (pre-pass, attention, merge of split pairs).
 */
size_t pa_decode_multi_workspace_bytes(const pa_shape* shape, int32_t max_q_len);

pa_status pa_decode_multi(const pa_shape* shape, int32_t max_q_len, int32_t total_q, const void* q,
                          const int32_t* q_start, const void* k_pool, const void* v_pool,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          void* out, void* workspace, size_t workspace_bytes, uint32_t* err_word,
                          void* stream);

/*
 * 8-bit (FP8) KV cache.  Storing keys and values in 8 bits halves the cache
 * (ontq "AI Inference Serving at Scale", section 6; the vLLM deployment
 * script on thewebvale, section 5, names fp8_e5m2 as a cache dtype).
 * kv_format: PA_FP8_E4M3 (OCP E4M3, largest 448, no infinities) or
 * PA_FP8_E5M2.  The cache stores code(x / scale) with one fp32 scale for K
 * (k_scale) and one for V (v_scale), rounded to nearest even and saturated.
 * Layout: ONE pool of bytes [NB][Hkv][2][B * d]; each (block, KV head) piece
 * holds its B K rows ([B][d]) and then its V dims-first ([d][B]), so a piece
 * is one contiguous 2 * B * d bytes.  Within K row r the sixteen-byte parts
 * are permuted: part c (dims 16c .. 16c + 15) sits at part position
 * c XOR (r mod 8); the row keeps its own 128 bytes.  Supported: head_dim 128, B in {16, 32},
 * g in {1, 2, 4, 8, 16}, q and out fp16/bf16.
 *
 * pa_append_kv_fp8: quantize k_new / v_new (shape->dtype, [T][Hkv][d]) into
 * the pool at slot_mapping (negative skips; past the pool: PA_DEVERR_SLOT).
 * pa_decode_fp8: pa_decode over the 8-bit pool, i.e. attention over
 * K = k_scale * decode(code), V = v_scale * decode(code).  It computes in fp16
 * on the tensor cores: q is rounded to fp16 (exact inside fp16's normal
 * range; a bf16 query beyond fp16's finite range sets PA_DEVERR_Q_RANGE),
 * codes convert to fp16 exactly, accumulation is fp32.  Its workspace is sized
 * by pa_decode_fp8_workspace_bytes.
 * pa_copy_blocks_fp8: copy-on-write copies of whole blocks (all pieces) of
 * the 8-bit pool, as pa_copy_blocks; shape->dtype is the pool's kv_format.
 */
size_t pa_decode_fp8_workspace_bytes(const pa_shape* shape, int32_t kv_format);

pa_status pa_decode_fp8(const pa_shape* shape, int32_t kv_format, const void* q, const void* kv_pool,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        float k_scale, float v_scale, void* out, void* workspace,
                        size_t workspace_bytes, uint32_t* err_word, void* stream);

pa_status pa_append_kv_fp8(const pa_shape* shape, int32_t kv_format, int32_t num_tokens,
                           const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           void* kv_pool, float k_scale, float v_scale, uint32_t* err_word,
                           void* stream);

pa_status pa_copy_blocks_fp8(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs,
                             void* kv_pool, uint32_t* err_word, void* stream);

/*
 * Prefix-aware paged decode: the same results as pa_decode (up to rounding
 * order), with the leading blocks that a group of sequences shares read once
 * for the whole group.  Parallel samples of one prompt and requests behind a
 * common system prompt point at the same physical prompt blocks (ontq
 * section 3, "Copy-on-Write Memory Sharing"; letsbuildsolutions,
 * "Production Considerations", prefix caching; thewebvale section 2).
 *
 *   num_groups           groups of sequences (0: plain decode)
 *   group_starts         device int32 [num_groups + 1], ascending: group i is
 *                        sequences [group_starts[i], group_starts[i + 1])
 *   group_prefix_blocks  device int32 [num_groups]: every member of group i has
 *                        the same first group_prefix_blocks[i] table entries
 *                        and at least that many full blocks of context
 * Sequences outside every group are decoded as by pa_decode.  The kernel
 * checks the claim: a member whose table or length breaks it, or a malformed
 * group description, sets PA_DEVERR_GROUP and the affected rows are NaN (a
 * malformed group is treated as having no prefix); no access leaves the
 * tables, pools or workspace.  On `stream`: a memset of the workspace's
 * counters, the prefix pass (one (group, KV head) item reads the shared
 * blocks for up to 32 query rows), then the decode's pre-pass, attention
 * kernel and merge over each sequence's own blocks, the attention kernel
 * folding the prefix state in by the log-sum-exp rule.  Workspace: see
 * pa_decode_shared_prefix_workspace_bytes (no initialisation needed).
 */
size_t pa_decode_shared_prefix_workspace_bytes(const pa_shape* shape);

pa_status pa_decode_shared_prefix(const pa_shape* shape, const void* q, const void* k_pool,
                                  const void* v_pool, const int32_t* block_tables,
                                  const int32_t* context_lens, int32_t num_groups,
                                  const int32_t* group_starts, const int32_t* group_prefix_blocks,
                                  float scale, void* out, void* workspace, size_t workspace_bytes,
                                  uint32_t* err_word, void* stream);

/*
 * Append new tokens' keys and values to the cache (ontq section 3, on-demand
 * allocation; thewebvale section 2, block table).  For i < num_tokens with
 * slot = slot_mapping[i] >= 0:
 *     k_pool[slot / B][kh][slot % B][:] = k_new[i][kh][:]   for every kh (same for V)
 * A negative slot skips the row.  Bit-exact copy.  Two live rows with the same
 * slot in one call race (the block manager never emits that).
 *
 *   k_new, v_new  [num_tokens][Hkv][d]
 *   slot_mapping  int64 [num_tokens]
 * Uses shape->num_kv_heads, head_dim, block_size, num_blocks, dtype.
 */
pa_status pa_append_kv(const pa_shape* shape, int32_t num_tokens, const void* k_new,
                       const void* v_new, const int64_t* slot_mapping, void* k_pool,
                       void* v_pool, uint32_t* err_word, void* stream);

/*
 * Copy-on-write block copies (ontq section 3, "Copy-on-Write Memory
 * Sharing": only the diverged block is copied; thewebvale section 2).  For each
 * pair (src, dst) = (pairs[2i], pairs[2i+1]), i < num_pairs, the whole block
 * (every KV head and slot, K and V) of src is copied to dst.  Bit-exact.  A dst
 * must not appear twice or as a src in the same call (the block manager
 * always copies into a freshly taken block); src == dst is a no-op.
 *
 *   src_dst_pairs int32 [num_pairs][2] (device)
 */
pa_status pa_copy_blocks(const pa_shape* shape, const int32_t* src_dst_pairs, int32_t num_pairs,
                         void* k_pool, void* v_pool, uint32_t* err_word, void* stream);

/*
 * Paged decode attention without caller-provided scratch -- no counterpart on
 * the pages; it exists for callers that cannot allocate device memory (a host
 * framework that has reserved the device's memory for its own pool, a plugin
 * host that passes only inputs and outputs, a serving loop that must not call
 * cudaMalloc/cudaFree because they may synchronise the device).
 *
 * Same arguments and results as pa_decode, minus the workspace: the scratch is
 * a static device buffer of PA_NOALLOC_SCRATCH_BYTES inside the library, held
 * on every GPU that loads it until the process exits.  This call allocates
 * nothing.
 *  - Shapes whose minimum scratch exceeds PA_NOALLOC_SCRATCH_BYTES are
 *    rejected with PA_ERR_WORKSPACE before anything is enqueued; shapes whose
 *    preferred scratch exceeds it run with fewer run-time balanced chunks.
 *  - Every call looks up the buffer's address on the current device (a failed
 *    lookup returns PA_ERR_CUDA).  The first lookup on a device may load the
 *    library's device code; make the first call on each device before any
 *    stream capture.
 *  - Every call on a device shares the one buffer and it keeps the last call's
 *    contents (the call clears the part that must start at zero).  Calls that
 *    overlap on the GPU -- on different streams, or unordered from different
 *    threads -- race on it and give wrong results; order them on one stream.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

pa_status pa_decode_noalloc(const pa_shape* shape, const void* q, const void* k_pool,
                            const void* v_pool, const int32_t* block_tables,
                            const int32_t* context_lens, float scale, void* out,
                            uint32_t* err_word, void* stream);

/*
 * Fault injection for tests of the wait limit (no counterpart on the pages).
 * With wait_ns > 0, every later launch of the decode attention kernel (by
 * pa_decode, pa_decode_noalloc, pa_decode_fp8, pa_decode_int4 and the second
 * pass of pa_decode_shared_prefix), in any thread of the process, makes each
 * worker warp's first stage wait on a shared-memory barrier that nothing
 * completes, for at most wait_ns.  When it gives up, the kernel takes its
 * timeout path: it sets PA_DEVERR_TIMEOUT, issues no further copies, writes
 * NaN to every output row and partial state of that worker, waits (at the
 * normal 2 s limit) for its copies still in flight and returns.  The call's
 * outputs are then NaN (rows of zero-length contexts stay zero) and
 * pa_read_error returns PA_ERR_TIMEOUT.  wait_ns = 0 turns it off (the
 * default).  wait_ns above 1e9 (1 s): PA_ERR_INVALID_ARG.
 */
pa_status pa_set_decode_stall_ns(uint64_t wait_ns);

/*
 * Synchronise `stream`, read the device error word and map it to a status:
 * PA_ERR_TIMEOUT if the timeout bit is set, else PA_ERR_OUT_OF_RANGE if any
 * other bit is set, else PA_OK.  The word is left unchanged.
 */
pa_status pa_read_error(const uint32_t* err_word, void* stream);

/* Static description of a status code. */
const char* pa_status_string(pa_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
