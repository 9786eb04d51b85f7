// Instantiations of the prefix pass of prefix-aware decode.
#include "prefix_kernel.cuh"

namespace pa {

void prefix_table(PrefixKernelInfo (&t)[2][2][2]) {
    t[0][0][0] = prefix_info<PrefixTraits<64, 16, false>>();
    t[0][0][1] = prefix_info<PrefixTraits<64, 32, false>>();
    t[0][1][0] = prefix_info<PrefixTraits<128, 16, false>>();
    t[0][1][1] = prefix_info<PrefixTraits<128, 32, false>>();
    t[1][0][0] = prefix_info<PrefixTraits<64, 16, true>>();
    t[1][0][1] = prefix_info<PrefixTraits<64, 32, true>>();
    t[1][1][0] = prefix_info<PrefixTraits<128, 16, true>>();
    t[1][1][1] = prefix_info<PrefixTraits<128, 32, true>>();
}

}  // namespace pa
