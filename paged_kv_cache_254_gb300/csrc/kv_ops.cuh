// Launch interface of the append and block-copy kernels (kv_ops.cu).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace pa {

struct AppendArgs {
    int32_t T;             // rows of k_new / v_new
    int32_t Hkv;
    int32_t vec_per_row;   // head_dim * 2 / 16
    int32_t BS;
    long long num_slots;   // num_blocks * block_size
    uint32_t* err;
};

struct CopyArgs {
    long long n;              // pairs
    long long vec_per_block;  // Hkv * BS * head_dim * 2 / 16
    int32_t NB;
    uint32_t* err;
};

struct Append8Args {
    int32_t T, Hkv, D, BS;
    long long num_slots;
    float k_scale, v_scale;
    uint32_t* err;
};

struct Append4Args {
    int32_t T, Hkv, BS;
    int32_t piece_bytes;   // bytes of one (block, head) piece
    long long num_slots;
    uint32_t* err;
};

cudaError_t append4_launch(const void* k_new, const void* v_new, const int64_t* slots, void* kv_pool,
                           const Append4Args& a, bool bf16, cudaStream_t stream, int sms);
cudaError_t append8_launch(const void* k_new, const void* v_new, const int64_t* slots, void* kv_pool,
                           const Append8Args& a, bool bf16, bool e5m2, cudaStream_t stream, int sms);
cudaError_t append_launch(const void* k_new, const void* v_new, const int64_t* slots, void* k_pool,
                          void* v_pool, const AppendArgs& a, cudaStream_t stream, int sms);
cudaError_t copy_launch(const int32_t* pairs, void* k_pool, void* v_pool, const CopyArgs& a,
                        cudaStream_t stream, int sms);

}  // namespace pa
