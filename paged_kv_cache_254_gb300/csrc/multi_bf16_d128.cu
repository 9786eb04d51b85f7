// Instantiations of the multi-token query kernel: bf16, head_dim 128.
#include "multi_kernel.cuh"

namespace pa {

void multi_table_bf16_d128(MultiKernelInfo (&t)[2][4]) {
    t[0][0] = multi_info<MultiTraits<128, 16, 1, true>>();
    t[0][1] = multi_info<MultiTraits<128, 16, 2, true>>();
    t[0][2] = multi_info<MultiTraits<128, 16, 4, true>>();
    t[0][3] = multi_info<MultiTraits<128, 16, 8, true>>();
    t[1][0] = multi_info<MultiTraits<128, 32, 1, true>>();
    t[1][1] = multi_info<MultiTraits<128, 32, 2, true>>();
    t[1][2] = multi_info<MultiTraits<128, 32, 4, true>>();
    t[1][3] = multi_info<MultiTraits<128, 32, 8, true>>();
}

}  // namespace pa
