// Real spherical harmonics of edge vectors, degrees 0..3, "component"
// normalisation (sum_m Y_lm^2 = 2l+1 on unit vectors), real basis m = -l..l
// with z as pole and no Condon-Shortley sign ("cuEquivariance in PyTorch",
// Spherical harmonics and a NumPy reference; Lesson 12a, section 21.5).
//
// Written as the harmonic homogeneous polynomials of degree l in (x, y, z)
// (the solid harmonics r^l Y_lm), obtained from the Cartesian forms of the
// real harmonics times sqrt(4 pi):
//   l=1: sqrt(3) (y, z, x)
//   l=2: sqrt(15) xy, sqrt(15) yz, sqrt(5)/2 (2z^2-x^2-y^2), sqrt(15) xz, sqrt(15)/2 (x^2-y^2)
//   l=3: sqrt(70)/4 y(3x^2-y^2), sqrt(105) xyz, sqrt(42)/4 y(4z^2-x^2-y^2),
//        sqrt(7)/2 z(2z^2-3x^2-3y^2), sqrt(42)/4 x(4z^2-x^2-y^2),
//        sqrt(105)/2 z(x^2-y^2), sqrt(70)/4 x(x^2-3y^2)
// With normalize != 0 the vector is first scaled to unit length, so these are
// the harmonics of the direction.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace tpc {

struct ShParams {
    const float *vec;
    float *sh;
    int64_t n;
    int32_t dim_sh;
    int32_t n_blocks;
    int32_t normalize;
    uint8_t l[kMaxShBlocks];
};

__global__ void sh_kernel(const __grid_constant__ ShParams P) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= P.n) return;
    float x = P.vec[3 * e + 0], y = P.vec[3 * e + 1], z = P.vec[3 * e + 2];
    if (P.normalize) {
        const float r2 = x * x + y * y + z * z;
        const float inv = r2 > 0.f ? rsqrtf(r2) : 0.f;
        x *= inv;
        y *= inv;
        z *= inv;
    }
    float Y[16];
    const float x2 = x * x, y2 = y * y, z2 = z * z;
    Y[0] = 1.f;
    const float s3 = 1.7320508075688772f;
    Y[1] = s3 * y;
    Y[2] = s3 * z;
    Y[3] = s3 * x;
    const float s15 = 3.872983346207417f, s5h = 1.118033988749895f;
    Y[4] = s15 * x * y;
    Y[5] = s15 * y * z;
    Y[6] = s5h * (2.f * z2 - x2 - y2);
    Y[7] = s15 * x * z;
    Y[8] = 0.5f * s15 * (x2 - y2);
    const float c70 = 2.0916500663351889f;   // sqrt(70)/4
    const float c105 = 10.246950765959598f;  // sqrt(105)
    const float c42 = 1.6201851746019651f;   // sqrt(42)/4
    const float c7 = 1.3228756555322954f;    // sqrt(7)/2
    Y[9] = c70 * y * (3.f * x2 - y2);
    Y[10] = c105 * x * y * z;
    Y[11] = c42 * y * (4.f * z2 - x2 - y2);
    Y[12] = c7 * z * (2.f * z2 - 3.f * x2 - 3.f * y2);
    Y[13] = c42 * x * (4.f * z2 - x2 - y2);
    Y[14] = 0.5f * c105 * z * (x2 - y2);
    Y[15] = c70 * x * (x2 - 3.f * y2);
    float *out = P.sh + e * P.dim_sh;
    int o = 0;
    for (int b = 0; b < P.n_blocks; ++b) {
        const int l = P.l[b];
        for (int m = 0; m < 2 * l + 1; ++m) out[o + m] = Y[l * l + m];
        o += 2 * l + 1;
    }
}

cudaError_t sh_launch(const float *vec, int64_t E, int normalize, const Tables &T, float *sh, cudaStream_t stream) {
    if (E == 0) return cudaSuccess;
    ShParams P;
    P.vec = vec;
    P.sh = sh;
    P.n = E;
    P.dim_sh = T.dim_sh;
    P.n_blocks = T.n_sh_blocks;
    P.normalize = normalize;
    for (int b = 0; b < kMaxShBlocks; ++b) P.l[b] = b < T.n_sh_blocks ? T.sh_l[b] : 0;
    const int threads = 256;
    const int64_t blocks = (E + threads - 1) / threads;
    sh_kernel<<<(unsigned)blocks, threads, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace tpc
