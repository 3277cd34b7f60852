// Conversions around the fused forward for tp_conv_forward_ex and
// tp_transpose_layout: int64 -> int32 indices, blockwise mul_ir <-> ir_mul row
// layouts (Lesson 12a, section 21.3), and the mean over a destination's edges.
// Each is one pass streaming its rows through HBM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace tpc {

__global__ void indices_to_i32_kernel(const int64_t *__restrict__ in, int64_t n, int32_t *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t v = in[i];
        out[i] = (v < 0 || v > 0x7fffffffll) ? -1 : (int32_t)v;
    }
}

cudaError_t indices_to_i32(const int64_t *in, int64_t n, int32_t *out, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    indices_to_i32_kernel<<<(unsigned)(blocks < 65536 ? blocks : 65536), 256, 0, stream>>>(in, n, out);
    return cudaGetLastError();
}

struct LayoutBlocks {
    int32_t n, dim;
    int32_t off[8], mul[8], ir[8];  // block offset, multiplicity, 2l+1
};

// Element (mu, i) of block b sits at off + mu*ir + i in mul_ir and at
// off + i*mul + mu in ir_mul. One thread per destination element.
template <typename T>
__global__ void transpose_rows_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t rows,
                                      const LayoutBlocks B, int to_ir_mul) {
    const int64_t total = rows * B.dim;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / B.dim;
        const int c = (int)(t - r * B.dim);
        int b = 0;
        while (b + 1 < B.n && c >= B.off[b + 1]) ++b;
        const int q = c - B.off[b], mul = B.mul[b], ir = B.ir[b];
        int sq;
        if (to_ir_mul) {  // dst (i, mu) at q = i*mul + mu; src at mu*ir + i
            const int i = q / mul, mu = q - i * mul;
            sq = mu * ir + i;
        } else {  // dst (mu, i) at q = mu*ir + i; src at i*mul + mu
            const int mu = q / ir, i = q - mu * ir;
            sq = i * mul + mu;
        }
        dst[t] = src[r * B.dim + B.off[b] + sq];
    }
}

cudaError_t transpose_rows(const tp_desc *d, int which, int from, const void *src, void *dst, int64_t rows,
                           int elem_bytes, cudaStream_t stream) {
    LayoutBlocks B;
    B.n = which == 0 ? d->n_in : d->n_out;
    B.dim = which == 0 ? d->tab.dim_x : d->tab.dim_out;
    for (int b = 0; b < B.n; ++b) {
        B.off[b] = which == 0 ? d->in_off[b] : d->out_off[b];
        B.mul[b] = which == 0 ? d->in_mul[b] : d->out_mul[b];
        B.ir[b] = 2 * (which == 0 ? d->in_l[b] : d->out_l[b]) + 1;
    }
    const int64_t total = rows * B.dim;
    if (total <= 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    const unsigned g = (unsigned)(blocks < 1048576 ? blocks : 1048576);
    const int to_ir = from == TP_MUL_IR;
    if (elem_bytes == 4)
        transpose_rows_kernel<uint32_t><<<g, 256, 0, stream>>>(static_cast<const uint32_t *>(src),
                                                               static_cast<uint32_t *>(dst), rows, B, to_ir);
    else
        transpose_rows_kernel<uint16_t><<<g, 256, 0, stream>>>(static_cast<const uint16_t *>(src),
                                                               static_cast<uint16_t *>(dst), rows, B, to_ir);
    return cudaGetLastError();
}

// out[d, :] /= (row_ptr[d+1] - row_ptr[d]) for destinations with edges; one
// warp per row, 16-byte accesses (dim is a multiple of 4).
__global__ void scale_rows_kernel(float *__restrict__ out, const int32_t *__restrict__ row_ptr, int32_t n, int32_t dim) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= n) return;
    const int deg = row_ptr[warp + 1] - row_ptr[warp];
    if (deg <= 1) return;  // empty rows are zero already; one edge: the mean is the sum
    const float inv = 1.f / (float)deg;
    float4 *row = reinterpret_cast<float4 *>(out + warp * dim);
    for (int c = lane; c < dim / 4; c += 32) {
        float4 v = row[c];
        v.x *= inv;
        v.y *= inv;
        v.z *= inv;
        v.w *= inv;
        row[c] = v;
    }
}

cudaError_t scale_rows_by_inverse_degree(float *out, const int32_t *row_ptr, int32_t n, int32_t dim,
                                         cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = ((int64_t)n * 32 + 255) / 256;
    scale_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out, row_ptr, n, dim);
    return cudaGetLastError();
}

}  // namespace tpc
