// Instantiations of the direct-load forward kernel, __nv_bfloat16 inputs
// (bfloat16 rows are copied as 4-byte pairs, so two or more channels per lane).
#include "direct_fwd.cuh"

namespace tpc {

const void *direct_kernel_bf16(int shape, int cpt) {
#define TPC_D(SI, LI, LSH, LO) \
    if (shape == SI && cpt == 2) return reinterpret_cast<const void *>(&direct_fwd_kernel<LI, LSH, LO, 2, __nv_bfloat16>);
    TPC_D(0, 1, 1, 1) TPC_D(1, 1, 2, 2) TPC_D(2, 2, 3, 2) TPC_D(3, 3, 3, 3)
#undef TPC_D
    return nullptr;
}

}  // namespace tpc
