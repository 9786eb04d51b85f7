// Instantiations of the multi-token query kernel: fp16, head_dim 128.
#include "multi_kernel.cuh"

namespace pa {

void multi_table_fp16_d128(MultiKernelInfo (&t)[2]) {
    t[0] = multi_info<MultiTraits<128, 16, 1, false>>();
    t[1] = multi_info<MultiTraits<128, 32, 1, false>>();
}

}  // namespace pa
