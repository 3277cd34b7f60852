"""fp64 CPU oracle for the fused equivariant tensor-product convolution.

TEST INFRASTRUCTURE ONLY. Nothing in the library (the CUDA path, its C ABI or
its Python binding) imports, links or runs anything in this package. Only the
test-suite, the smoke check and the CPU-baseline leg of the benchmark use it.

It is a plain, slow, obviously correct restatement of what the method computes,
in float64, written independently of the CUDA path (no shared code, tables or
generators):

* ``irreps``   irreps strings, dimensions and the two block layouts
               (Lesson 12a: Foundations of cuEquivariance, sections 21.2-21.3).
* ``so3``      real spherical harmonics from associated Legendre functions,
               rotation matrices, Wigner-D matrices by least squares on the
               harmonics, and real Clebsch-Gordan tensors as the null space of
               the equivariance constraint (section 21.1: the coefficients are
               fixed by the group and mostly zero).
* ``tp``       path enumeration (section 21.4), the channelwise ``uvu``
               contraction ``[ijk]·a[uv]·b[iu]·c[jv] -> D[kuv]`` with per-edge
               weights, gather by source and sum-scatter to destination
               ("cuEquivariance in PyTorch", SegmentedPolynomial: gather and
               scatter), its exact (trilinear) backward, and the stable
               counting sort that defines the CSR.
* ``cref``     the same forward/backward as plain C loops with OpenMP, used for
               sizes the numpy version is too slow for and for the CPU baseline.

Readings of points the pages leave open:
real basis ordered m=-l..l with the z axis as pole and l=1 = sqrt(3)(y,z,x);
"component" normalisation (sum_m Y_lm^2 = 2l+1 on the unit sphere);
Clebsch-Gordan tensors orthonormal over (i,j) for each k with no extra path
factor, sign fixed so that the first nonzero entry in (i,j,k) row-major order
is positive; paths with the same output irrep type sum into that one output
block, in the order of the output irreps string.
"""
