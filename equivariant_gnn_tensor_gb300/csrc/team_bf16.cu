// Instantiations of the program-specialised forward kernel, __nv_bfloat16 inputs.
#include "team_fwd.cuh"

namespace tpc {

const void *team_kernel_bf16(int shape, int cpt) {
#define TPC_T(SI, LI, LSH, LO) \
    if (shape == SI && cpt == 1) return reinterpret_cast<const void *>(&team_fwd_kernel<LI, LSH, LO, 1, __nv_bfloat16>); \
    if (shape == SI && cpt == 2) return reinterpret_cast<const void *>(&team_fwd_kernel<LI, LSH, LO, 2, __nv_bfloat16>); \
    if (shape == SI && cpt == 4) return reinterpret_cast<const void *>(&team_fwd_kernel<LI, LSH, LO, 4, __nv_bfloat16>);
    TPC_T(0, 1, 1, 1) TPC_T(1, 1, 2, 2) TPC_T(2, 2, 3, 2) TPC_T(3, 3, 3, 3)
#undef TPC_T
    return nullptr;
}

}  // namespace tpc
