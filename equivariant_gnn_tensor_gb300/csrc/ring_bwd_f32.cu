// Instantiations of the backward ring kernel, float inputs.
#include "ring_bwd.cuh"

namespace tpc {

// cpt: channels per lane (mul = 32 * cpt); two or four channels per lane run
// as packed pairs.
const void *ring_bwd_kernel_f32(int shape, int cpt) {
#define TPC_R(SI, LI, LSH, LO) \
    if (shape == SI && cpt == 1) return reinterpret_cast<const void *>(&ring_bwd_kernel<LI, LSH, LO, 1, false, float>); \
    if (shape == SI && cpt == 2) return reinterpret_cast<const void *>(&ring_bwd_kernel<LI, LSH, LO, 2, true, float>); \
    if (shape == SI && cpt == 4) return reinterpret_cast<const void *>(&ring_bwd_kernel<LI, LSH, LO, 4, true, float>);
    TPC_R(0, 1, 1, 1) TPC_R(1, 1, 2, 2) TPC_R(2, 2, 3, 2) TPC_R(3, 3, 3, 3)
#undef TPC_R
    return nullptr;
}

}  // namespace tpc
