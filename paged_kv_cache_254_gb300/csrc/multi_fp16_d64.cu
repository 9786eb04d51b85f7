// Instantiations of the multi-token query kernel: fp16, head_dim 64.
#include "multi_kernel.cuh"

namespace pa {

void multi_table_fp16_d64(MultiKernelInfo (&t)[2]) {
    t[0] = multi_info<MultiTraits<64, 16, 1, false>>();
    t[1] = multi_info<MultiTraits<64, 32, 1, false>>();
}

}  // namespace pa
