// Forward with one output block per path (descriptors from
// tp_desc_create_unsimplified; Lesson 12a, section 21.4: the descriptor lists
// one output block per path). Each path's sum has a block of its own, so the
// per-destination row is wider than the register rows of the other kernels:
// one warp per destination accumulates it in shared memory (lane = channel,
// channels lane + 32c), gathering x and w rows straight from global memory
// (L1/L2), with M_p[i][k] = sum_j C_p[i,j,k] sh[b_p, j] built per edge from
// the descriptor's recipe. Fixed summation order, no atomics.
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"

namespace tpc {

struct UnsimpParams {
    Tables tab;
    int32_t out_off[kMaxPaths];  // output block of path p
    int32_t dim_u;               // output row width
    int32_t acc_floats;          // per-warp accumulator row (dim_u rounded)
    const void *x;
    const float *sh;
    const void *w;
    const int32_t *src, *row_ptr;
    float *out;
    int *status;
    int32_t n_src, n_dst;
    int64_t E;
};

constexpr int kUnsimpWarps = 4;

template <typename FT>
__device__ __forceinline__ float ld_elem(const FT *p) {
    if constexpr (sizeof(FT) == 4) return __ldg(reinterpret_cast<const float *>(p));
    else return __bfloat162float(*p);
}

template <typename FT>
__global__ void __launch_bounds__(32 * kUnsimpWarps) unsimp_fwd_kernel(const __grid_constant__ UnsimpParams prm) {
    extern __shared__ __align__(16) unsigned char smem[];
    const Tables &T = prm.tab;
    SmemTables *st = reinterpret_cast<SmemTables *>(smem);
    for (int q = threadIdx.x; q <= T.R; q += blockDim.x) st->rec_ptr[q] = T.rec_ptr[q];
    for (int q = threadIdx.x; q < T.nnz; q += blockDim.x) {
        st->rec_j[q] = T.rec_j[q];
        st->rec_c[q] = T.rec_c[q];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *acc = reinterpret_cast<float *>(smem + ((sizeof(SmemTables) + 15) / 16 * 16)) +
                 (size_t)warp * (prm.acc_floats + T.R + 64);
    float *M = acc + prm.acc_floats;
    float *shr = M + T.R;
    const FT *xp = static_cast<const FT *>(prm.x);
    const FT *wp = static_cast<const FT *>(prm.w);
    const int mul = T.mul;
    const int nw = gridDim.x * kUnsimpWarps;
    for (int d = blockIdx.x * kUnsimpWarps + warp; d < prm.n_dst; d += nw) {
        for (int q = lane; q < prm.dim_u; q += 32) acc[q] = 0.f;
        int e0 = prm.row_ptr[d], e1 = prm.row_ptr[d + 1];
        if (e0 < 0 || e1 < e0 || e1 > prm.E) {
            if (lane == 0) set_status(prm.status, TP_DEV_ERR_SEGMENT);
            e1 = e0;
        }
        __syncwarp();
        for (int e = e0; e < e1; ++e) {
            const int s = prm.src[e];
            if ((uint32_t)s >= (uint32_t)prm.n_src) {
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
                continue;
            }
            for (int j = lane; j < T.dim_sh; j += 32) shr[j] = prm.sh[(int64_t)e * T.dim_sh + j];
            __syncwarp();
            for (int r = lane; r < T.R; r += 32) {
                float v = 0.f;
                for (int t = st->rec_ptr[r]; t < st->rec_ptr[r + 1]; ++t) v = fmaf(st->rec_c[t], shr[st->rec_j[t]], v);
                M[r] = v;
            }
            __syncwarp();
            const FT *xrow = xp + (int64_t)s * T.dim_x;
            const FT *wrow = wp + (int64_t)e * T.wnum;
            for (int p = 0; p < T.n_paths; ++p) {
                const int la = T.la[p], lc = T.lc[p], na = 2 * la + 1, nc = 2 * lc + 1;
                const float *Mp = M + T.m_off[p];
                const int xo = T.x_off[la], oo = prm.out_off[p];
                for (int ch = lane; ch < mul; ch += 32) {
                    float xv[7];
                    for (int i = 0; i < na; ++i) xv[i] = ld_elem(xrow + xo + i * mul + ch);
                    const float wv = ld_elem(wrow + p * mul + ch);
                    for (int k = 0; k < nc; ++k) {
                        float t = 0.f;
                        for (int i = 0; i < na; ++i) t = fmaf(Mp[i * nc + k], xv[i], t);
                        acc[oo + k * mul + ch] = fmaf(wv, t, acc[oo + k * mul + ch]);
                    }
                }
            }
            __syncwarp();
        }
        float *orow = prm.out + (int64_t)d * prm.dim_u;
        for (int q = lane; q < prm.dim_u; q += 32) orow[q] = acc[q];
        __syncwarp();
    }
}

cudaError_t unsimp_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                           const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                           float *out, int sms, int smem_optin, int *status, cudaStream_t stream) {
    static_assert(sizeof(UnsimpParams) < 32000, "kernel parameter block too large");
    UnsimpParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.tab = d->tab;
    for (int p = 0; p < d->n_paths; ++p) prm.out_off[p] = d->unsimp_off[p];
    prm.dim_u = d->unsimp_dim_out;
    prm.acc_floats = (d->unsimp_dim_out + 3) / 4 * 4;
    prm.x = x;
    prm.sh = sh;
    prm.w = w;
    prm.src = src;
    prm.row_ptr = row_ptr;
    prm.out = out;
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.E = E;
    const size_t smem = (sizeof(SmemTables) + 15) / 16 * 16 +
                        (size_t)kUnsimpWarps * (prm.acc_floats + d->tab.R + 64) * sizeof(float);
    if (smem > (size_t)smem_optin) return cudaErrorNotSupported;
    const void *fn = dtype == TP_F32 ? reinterpret_cast<const void *>(&unsimp_fwd_kernel<float>)
                                     : reinterpret_cast<const void *>(&unsimp_fwd_kernel<__nv_bfloat16>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 32 * kUnsimpWarps, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    long long blocks = ((long long)N_dst + kUnsimpWarps - 1) / kUnsimpWarps;
    if (blocks > (long long)sms * occ) blocks = (long long)sms * occ;
    if (blocks < 1) blocks = 1;
    void *args[] = {&prm};
    return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(32 * kUnsimpWarps), args, smem, stream);
}

}  // namespace tpc
