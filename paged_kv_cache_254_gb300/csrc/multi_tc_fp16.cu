// Instantiations of the tensor-core multi-token query kernel: fp16.
#include "multi_tc_kernel.cuh"

namespace pa {

void multi_tc_table_fp16_d128(MultiKernelInfo (&t)[2]) {
    t[0] = multi_tc_info<TcTraits<128, 16, false>>();
    t[1] = multi_tc_info<TcTraits<128, 32, false>>();
}

void multi_tc_table_fp16_d64(MultiKernelInfo (&t)[2]) {
    t[0] = multi_tc_info<TcTraits<64, 16, false>>();
    t[1] = multi_tc_info<TcTraits<64, 32, false>>();
}

}  // namespace pa
