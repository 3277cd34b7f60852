// Host-side launch entry points of the kernel translation units.
#pragma once
#include <cuda_runtime.h>

#include "conv_seg.cuh"

namespace tpc {

// Covering kernel shape for (max input degree, max output degree): the
// register slots of every degree up to LI / LO exist; absent degrees idle.
struct Shape {
    int li, lo;
};
inline bool pick_shape(int lmax_in, int lmax_out, Shape &s) {
    static const Shape shapes[] = {{1, 2}, {2, 2}, {3, 3}};
    for (const Shape &c : shapes)
        if (lmax_in <= c.li && lmax_out <= c.lo) {
            s = c;
            return true;
        }
    return false;
}
inline int pick_cpt(int mul) { return mul <= 32 ? 1 : (mul <= 64 ? 2 : 4); }

// Returns the kernel function pointer for the variant (nullptr if none).
const void *seg_fwd_f32_kernel(Shape s, int cpt);
const void *seg_fwd_bf16_kernel(Shape s, int cpt);
const void *seg_bwdx_f32_kernel(Shape s, int cpt);
const void *seg_bwde_f32_kernel(Shape s, int cpt);

}  // namespace tpc
