// Instantiations of the direct-load forward kernel, float inputs.
#include "direct_fwd.cuh"

namespace tpc {

const void *direct_kernel_f32(int shape, int cpt) {
#define TPC_D(SI, LI, LSH, LO) \
    if (shape == SI && cpt == 1) return reinterpret_cast<const void *>(&direct_fwd_kernel<LI, LSH, LO, 1, float>); \
    if (shape == SI && cpt == 2) return reinterpret_cast<const void *>(&direct_fwd_kernel<LI, LSH, LO, 2, float>);
    TPC_D(0, 1, 1, 1) TPC_D(1, 1, 2, 2) TPC_D(2, 2, 3, 2) TPC_D(3, 3, 3, 3)
#undef TPC_D
    return nullptr;
}

}  // namespace tpc
