// Instantiations of the warp-ring forward kernel, edge-vector inputs with the weight rows computed by the radial network in the kernel, float inputs.
#include "ring_fwd.cuh"

namespace tpc {

// cpt: channels per lane (mul = 32 * cpt); pk: packed channel (cpt >= 2) or
// edge (cpt == 1) pairs. The register caps (blocks of 256 threads per SM) keep
// one channel per lane at 3 blocks per SM and packed pairs at 2; edge pairs of
// the two smaller programs form the weights in registers (a chunk's worth at
// once), at one block per SM.
const void *ring_kernel_mlp_f32(int shape, int cpt, int pk) {
#define TPC_R(SI, LI, LSH, LO, MINB_EP) \
    if (shape == SI && cpt == 1 && !pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 1, false, 3, float, 2>); \
    if (shape == SI && cpt == 1 && pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 1, true, MINB_EP, float, 2>); \
    if (shape == SI && cpt == 2 && !pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 2, false, 1, float, 2>); \
    if (shape == SI && cpt == 2 && pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 2, true, 2, float, 2>); \
    if (shape == SI && cpt == 4 && !pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 4, false, 1, float, 2>); \
    if (shape == SI && cpt == 4 && pk) return reinterpret_cast<const void *>(&ring_fwd_kernel<LI, LSH, LO, 4, true, 1, float, 2>);
    TPC_R(0, 1, 1, 1, 1) TPC_R(1, 1, 2, 2, 1) TPC_R(2, 2, 3, 2, 2) TPC_R(3, 3, 3, 3, 2)
#undef TPC_R
    return nullptr;
}

}  // namespace tpc
