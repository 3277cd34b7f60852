// Real spherical harmonics of edge vectors, degrees 0..3 (real_sh_upto in
// common.cuh; "cuEquivariance in PyTorch", Spherical harmonics and a NumPy
// reference; Lesson 12a, section 21.5), written out block by block in the
// order of the descriptor's harmonic irreps.
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
    float Y[16];
    real_sh_upto<3>(P.vec[3 * e + 0], P.vec[3 * e + 1], P.vec[3 * e + 2], P.normalize != 0, Y);
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
