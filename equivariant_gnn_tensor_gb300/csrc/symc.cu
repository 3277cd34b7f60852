// Symmetric contraction kernel (tp_symmetric_contraction): per node a
// polynomial of degree <= 3 in the node's own features, channel by channel.
//
// A warp evaluates two nodes at a time, one per half-warp, each lane two
// adjacent channels as a packed f32x2 pair (channels 2c, 2c+1 for
// c = lane, lane + 16, ...). Every element's weights are staged in shared
// memory once per block (when they fit; otherwise they are read through
// L1/L2), and the node feature rows stream through a per-warp double buffer
// of cp.async copies, the next pair's rows in flight while this pair is
// evaluated. The basis sits in the kernel's parameter space as warp-uniform
// operations, grouped by output row and then by weight: an operation is
// {three feature offsets, coefficient} (degree < 3 products padded with a
// row of ones, so every operation is the same branch-free coef * b1 * b2 * b3)
// and a group sums its operations into u before adding a_q * u to the row.
// The row sum over groups is compensated (Kahan), and so is the sum inside a
// group when groups are long, so the rounding error stays that of a few
// operations however many entries a row has. HBM traffic: one read of x and
// of the element index, one write of out.
#include <cuda_runtime.h>

#include "common.cuh"
#include "symc.h"

namespace tpc {
namespace {

constexpr int kSymcWarps = 8;
constexpr int kSymcMaxRows = 64;     // output rows (sum of 2L+1 over output blocks)
constexpr int kSymcMaxGroups = 512;  // (row, weight) groups
constexpr int kSymcShortGroup = 8;   // groups up to this long sum without compensation

struct SymcOp {
    int16_t o1, o2, o3;  // feature offsets in channel pairs (component * mul / 2); D * mul / 2 is the row of ones
    int16_t pad;
    float coef;
};

struct SymcGroup {
    int16_t oq;   // weight offset in channel pairs (weight index * mul / 2)
    uint16_t t0;  // first operation; the group ends where the next one starts
};

struct SymcParams {
    const float *x;
    const float *weights;
    const int32_t *element;
    float *out;
    int *status;
    int32_t N, num_elements, mul, dim_in, rows_out, n_weights, w_in_smem;
    int32_t row_ptr[kSymcMaxRows + 1];  // groups of output row r: [row_ptr[r], row_ptr[r+1])
    SymcGroup groups[kSymcMaxGroups + 1];
    SymcOp ops[kSymcMaxEntries];
};

typedef unsigned long long f2;
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_splat(float v) {
    f2 d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(v));
    return d;
}
// s + a * b with s, c the running Kahan sum and its (negated) lost low part
__device__ __forceinline__ void kahan_fma(f2 &s, f2 &nc, f2 a, f2 b) {
    const f2 y = f2_fma(a, b, nc);  // a * b - c
    const f2 t = f2_add(s, y);
    nc = f2_sub(y, f2_sub(t, s));   // -((t - s) - y)
    s = t;
}

template <bool KI>
__global__ void symc_kernel(const __grid_constant__ SymcParams P) {
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, hl = lane & 15, side = lane >> 4;
    const int wel_n = P.n_weights * P.mul;  // weights of one element
    const int row_n = P.dim_in + P.mul;     // staged row: features, then a row of ones
    float *wsm = sm;
    float *buf = sm + (P.w_in_smem ? (P.num_elements * wel_n + 3) / 4 * 4 : 0) + (size_t)warp * 4 * row_n;
    if (P.w_in_smem)
        for (int q = threadIdx.x; q < P.num_elements * wel_n; q += blockDim.x) wsm[q] = __ldg(P.weights + q);
    for (int k = 0; k < 4; ++k)
        for (int q = lane; q < P.mul; q += 32) buf[k * row_n + P.dim_in + q] = 1.f;
    __syncthreads();
    const int n4 = P.dim_in / 4, m2 = P.mul / 2;
    const int64_t stride = 2ll * gridDim.x * kSymcWarps;
    int64_t n = 2ll * (blockIdx.x * kSymcWarps + warp);
    // half-warp `side` stages node n + side into slot (it & 1) * 2 + side
#define SYMC_FETCH(n_, it_)                                                                  \
    do {                                                                                     \
        if ((n_) + side < P.N) {                                                             \
            const float *src_ = P.x + ((n_) + side) * P.dim_in;                              \
            float *dst_ = buf + (((it_) & 1) * 2 + side) * row_n;                            \
            for (int q_ = hl; q_ < n4; q_ += 16) cp_async16(dst_ + 4 * q_, src_ + 4 * q_);  \
        }                                                                                    \
        cp_async_commit();                                                                   \
    } while (0)
    SYMC_FETCH(n, 0);
    int el_next = n + side < P.N ? __ldg(P.element + n + side) : 0;
    for (int it = 0; n < P.N; n += stride, ++it) {
        const int64_t node = n + side;
        const f2 *b = reinterpret_cast<const f2 *>(buf + ((it & 1) * 2 + side) * row_n);
        const int el = el_next;
        SYMC_FETCH(n + stride, it + 1);
        el_next = n + stride + side < P.N ? __ldg(P.element + n + stride + side) : 0;
        const bool live = node < P.N;
        const bool ok = (uint32_t)el < (uint32_t)P.num_elements;
        if (live && !ok) set_status(P.status, TP_DEV_ERR_INDEX);
        const f2 *wel = reinterpret_cast<const f2 *>((P.w_in_smem ? wsm : P.weights) + (int64_t)(ok ? el : 0) * wel_n);
        cp_async_wait_pending(1);  // this pair's rows have landed
        __syncwarp();
        f2 *orow = reinterpret_cast<f2 *>(P.out + node * P.rows_out * P.mul);
        for (int c = hl; c < m2; c += 16) {
            const f2 *bc = b + c;
            const f2 *wc = wel + c;
            for (int r = 0; r < P.rows_out; ++r) {
                f2 acc = 0, nc = 0;
                for (int g = P.row_ptr[r]; g < P.row_ptr[r + 1]; ++g) {
                    const SymcGroup G = P.groups[g];
                    const int t1 = P.groups[g + 1].t0;
                    f2 u = 0, unc = 0;
                    for (int t = G.t0; t < t1; ++t) {
                        const SymcOp e = P.ops[t];
                        const f2 m = f2_mul(f2_mul(bc[e.o1], bc[e.o2]), bc[e.o3]);
                        if (KI)
                            kahan_fma(u, unc, f2_splat(e.coef), m);
                        else
                            u = f2_fma(f2_splat(e.coef), m, u);
                    }
                    kahan_fma(acc, nc, wc[G.oq], u);
                }
                if (live) orow[r * m2 + c] = ok ? acc : 0ull;
            }
        }
        __syncwarp();  // the buffer is refilled two pairs later
    }
    cp_async_wait_pending(0);
#undef SYMC_FETCH
}

}  // namespace

cudaError_t symc_launch(const tp_symc *s, const float *x, const float *weights, const int32_t *element, int32_t N,
                        int32_t num_elements, float *out, int sms, int smem_optin, int *status, cudaStream_t stream) {
    static_assert(sizeof(SymcParams) < 32000, "kernel parameter block too large");
    int n_entries = 0;
    const SymcEntry *tab = symc_table(s, &n_entries);
    SymcParams P;
    P.x = x;
    P.weights = weights;
    P.element = element;
    P.out = out;
    P.status = status;
    P.N = N;
    P.num_elements = num_elements;
    P.mul = symc_mul(s);
    const int D = symc_D(s);
    P.dim_in = D * P.mul;
    P.rows_out = symc_rows_out(s);
    P.n_weights = symc_n_weights(s);
    if (P.rows_out > kSymcMaxRows || (D + 1) * P.mul / 2 > 32767 || P.n_weights * P.mul / 2 > 32767)
        return cudaErrorNotSupported;
    // entries are grouped by output row, then by weight
    int n_groups = 0, longest = 0;
    for (int t = 0, r = 0; r < P.rows_out; ++r) {
        P.row_ptr[r] = n_groups;
        while (t < n_entries && tab[t].row == r) {
            if (n_groups == kSymcMaxGroups) return cudaErrorNotSupported;
            const int q = tab[t].q, t0 = t;
            P.groups[n_groups].oq = (int16_t)(q * P.mul / 2);
            P.groups[n_groups].t0 = (uint16_t)t;
            for (; t < n_entries && tab[t].row == r && tab[t].q == q; ++t) {
                const SymcEntry &e = tab[t];
                SymcOp &o = P.ops[t];
                o.o1 = (int16_t)(e.i1 * P.mul / 2);
                o.o2 = (int16_t)((e.nu >= 2 ? e.i2 : D) * P.mul / 2);
                o.o3 = (int16_t)((e.nu >= 3 ? e.i3 : D) * P.mul / 2);
                o.pad = 0;
                o.coef = e.coef;
            }
            longest = t - t0 > longest ? t - t0 : longest;
            ++n_groups;
        }
    }
    P.row_ptr[P.rows_out] = n_groups;
    P.groups[n_groups].oq = 0;
    P.groups[n_groups].t0 = (uint16_t)n_entries;
    const size_t rows_bytes = (size_t)kSymcWarps * 4 * (P.dim_in + P.mul) * sizeof(float);
    const size_t w_bytes = ((size_t)num_elements * P.n_weights * P.mul + 3) / 4 * 4 * sizeof(float);
    // all elements' weights in shared memory when that still leaves room for two blocks per SM
    P.w_in_smem = 2 * (rows_bytes + w_bytes) <= (size_t)smem_optin;
    const size_t smem = rows_bytes + (P.w_in_smem ? w_bytes : 0);
    if (smem > (size_t)smem_optin) return cudaErrorNotSupported;
    const void *fn = longest > kSymcShortGroup ? (const void *)symc_kernel<true> : (const void *)symc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 32 * kSymcWarps, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    long long blocks = ((long long)N + 2 * kSymcWarps - 1) / (2 * kSymcWarps);
    if (blocks > (long long)sms * occ) blocks = (long long)sms * occ;
    if (blocks < 1) blocks = 1;
    void *args[] = {&P};
    e = cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(32 * kSymcWarps), args, smem, stream);
    return e;
}

}  // namespace tpc
