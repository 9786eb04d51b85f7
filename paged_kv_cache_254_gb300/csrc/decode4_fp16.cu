// Instantiations of the decode kernel over the 4-bit cache, fp16 queries.
#include "decode_kernel.cuh"

namespace pa {

void decode4_table_fp16(DecodeKernelInfo (&t)[2][5]) {
    t[0][0] = decode_info<DecodeTraits<128, 16, 1, false, 3>>();
    t[0][1] = decode_info<DecodeTraits<128, 16, 2, false, 3>>();
    t[0][2] = decode_info<DecodeTraits<128, 16, 4, false, 3>>();
    t[0][3] = decode_info<DecodeTraits<128, 16, 8, false, 3>>();
    t[0][4] = decode_info<DecodeTraits<128, 16, 16, false, 3>>();
    t[1][0] = decode_info<DecodeTraits<128, 32, 1, false, 3>>();
    t[1][1] = decode_info<DecodeTraits<128, 32, 2, false, 3>>();
    t[1][2] = decode_info<DecodeTraits<128, 32, 4, false, 3>>();
    t[1][3] = decode_info<DecodeTraits<128, 32, 8, false, 3>>();
    t[1][4] = decode_info<DecodeTraits<128, 32, 16, false, 3>>();
}

}  // namespace pa
