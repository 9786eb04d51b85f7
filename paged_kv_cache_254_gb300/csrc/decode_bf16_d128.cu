// Instantiations of the paged decode kernel for bf16, head_dim 128.
#include "decode_kernel.cuh"

namespace pa {

void decode_table_bf16_d128(DecodeKernelInfo (&t)[2][5]) {
    t[0][0] = decode_info<DecodeTraits<128, 16, 1, true>>();
    t[0][1] = decode_info<DecodeTraits<128, 16, 2, true>>();
    t[0][2] = decode_info<DecodeTraits<128, 16, 4, true>>();
    t[0][3] = decode_info<DecodeTraits<128, 16, 8, true>>();
    t[0][4] = decode_info<DecodeTraits<128, 16, 16, true>>();
    t[1][0] = decode_info<DecodeTraits<128, 32, 1, true>>();
    t[1][1] = decode_info<DecodeTraits<128, 32, 2, true>>();
    t[1][2] = decode_info<DecodeTraits<128, 32, 4, true>>();
    t[1][3] = decode_info<DecodeTraits<128, 32, 8, true>>();
    t[1][4] = decode_info<DecodeTraits<128, 32, 16, true>>();
}

}  // namespace pa
