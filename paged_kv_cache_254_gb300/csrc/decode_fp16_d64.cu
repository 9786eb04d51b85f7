// Instantiations of the paged decode kernel for fp16, head_dim 64.
#include "decode_kernel.cuh"

namespace pa {

void decode_table_fp16_d64(DecodeKernelInfo (&t)[2][5]) {
    t[0][0] = decode_info<DecodeTraits<64, 16, 1, false>>();
    t[0][1] = decode_info<DecodeTraits<64, 16, 2, false>>();
    t[0][2] = decode_info<DecodeTraits<64, 16, 4, false>>();
    t[0][3] = decode_info<DecodeTraits<64, 16, 8, false>>();
    t[0][4] = decode_info<DecodeTraits<64, 16, 16, false>>();
    t[1][0] = decode_info<DecodeTraits<64, 32, 1, false>>();
    t[1][1] = decode_info<DecodeTraits<64, 32, 2, false>>();
    t[1][2] = decode_info<DecodeTraits<64, 32, 4, false>>();
    t[1][3] = decode_info<DecodeTraits<64, 32, 8, false>>();
    t[1][4] = decode_info<DecodeTraits<64, 32, 16, false>>();
}

}  // namespace pa
