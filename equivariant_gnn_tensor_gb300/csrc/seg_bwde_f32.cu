// Instantiations of the warp-per-segment kernel: mode kBwdEdge, feature type float.
#include "launch.h"

namespace tpc {

const void *seg_bwde_f32_kernel(Shape s, int cpt) {
#define TPC_K(LI, LO, C) \
    if (s.li == LI && s.lo == LO && cpt == C) return reinterpret_cast<const void *>(&seg_conv_kernel<LI, LO, C, float, kBwdEdge>);
    TPC_K(1, 2, 1) TPC_K(1, 2, 2) TPC_K(1, 2, 4)
    TPC_K(2, 2, 1) TPC_K(2, 2, 2) TPC_K(2, 2, 4)
    TPC_K(3, 3, 1) TPC_K(3, 3, 2) TPC_K(3, 3, 4)
#undef TPC_K
    return nullptr;
}

}  // namespace tpc
