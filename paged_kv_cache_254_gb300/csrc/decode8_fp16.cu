// Instantiations of the paged decode kernel over an 8-bit (FP8) cache, fp16 queries, head_dim 128.
#include "decode_kernel.cuh"

namespace pa {

void decode8_table_fp16(DecodeKernelInfo (&t)[2][2][5]) {
    t[0][0][0] = decode_info<DecodeTraits<128, 16, 1, false, 1>>();
    t[0][0][1] = decode_info<DecodeTraits<128, 16, 2, false, 1>>();
    t[0][0][2] = decode_info<DecodeTraits<128, 16, 4, false, 1>>();
    t[0][0][3] = decode_info<DecodeTraits<128, 16, 8, false, 1>>();
    t[0][0][4] = decode_info<DecodeTraits<128, 16, 16, false, 1>>();
    t[0][1][0] = decode_info<DecodeTraits<128, 32, 1, false, 1>>();
    t[0][1][1] = decode_info<DecodeTraits<128, 32, 2, false, 1>>();
    t[0][1][2] = decode_info<DecodeTraits<128, 32, 4, false, 1>>();
    t[0][1][3] = decode_info<DecodeTraits<128, 32, 8, false, 1>>();
    t[0][1][4] = decode_info<DecodeTraits<128, 32, 16, false, 1>>();
    t[1][0][0] = decode_info<DecodeTraits<128, 16, 1, false, 2>>();
    t[1][0][1] = decode_info<DecodeTraits<128, 16, 2, false, 2>>();
    t[1][0][2] = decode_info<DecodeTraits<128, 16, 4, false, 2>>();
    t[1][0][3] = decode_info<DecodeTraits<128, 16, 8, false, 2>>();
    t[1][0][4] = decode_info<DecodeTraits<128, 16, 16, false, 2>>();
    t[1][1][0] = decode_info<DecodeTraits<128, 32, 1, false, 2>>();
    t[1][1][1] = decode_info<DecodeTraits<128, 32, 2, false, 2>>();
    t[1][1][2] = decode_info<DecodeTraits<128, 32, 4, false, 2>>();
    t[1][1][3] = decode_info<DecodeTraits<128, 32, 8, false, 2>>();
    t[1][1][4] = decode_info<DecodeTraits<128, 32, 16, false, 2>>();
}

}  // namespace pa
