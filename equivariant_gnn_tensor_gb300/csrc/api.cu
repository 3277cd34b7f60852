// C-ABI entry points of libtpconv.so: argument checks, kernel selection,
// launch geometry and the per-device status word. See include/tpconv.h for
// the contract of every function.
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/tpconv.h"
#include "launch.h"
#include "tuning.h"

namespace tpc {
size_t csr_workspace_bytes(int64_t E, int32_t N);
cudaError_t csr_build_launch(const int32_t *keys, int64_t E, int32_t N, int32_t *perm, int32_t *row_ptr,
                             int32_t *keys_sorted, void *ws, int *status, cudaStream_t stream);
cudaError_t sh_launch(const float *vec, int64_t E, int normalize, const Tables &T, float *sh, cudaStream_t stream);
int64_t csr_noalloc_max_edges();
cudaError_t csr_noalloc_scratch(void **ptr);
size_t split_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin);
cudaError_t indices_to_i32(const int64_t *in, int64_t n, int32_t *out, cudaStream_t stream);
cudaError_t symc_jit_launch(const tp_symc *s, const float *x, const float *weights, const int32_t *element, int32_t N,
                            int32_t num_elements, float *out, int dev, int sms, int *status, cudaStream_t stream);
cudaError_t symc_launch(const tp_symc *s, const float *x, const float *weights, const int32_t *element, int32_t N,
                        int32_t num_elements, float *out, int sms, int smem_optin, int *status, cudaStream_t stream);
cudaError_t unsimp_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                           const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                           float *out, int sms, int smem_optin, int *status, cudaStream_t stream);
cudaError_t transpose_rows(const tp_desc *d, int which, int from, const void *src, void *dst, int64_t rows,
                           int elem_bytes, cudaStream_t stream);
cudaError_t scale_rows_by_inverse_degree(float *out, const int32_t *row_ptr, int32_t n, int32_t dim,
                                         cudaStream_t stream);
size_t mma_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin);
size_t ring_bwd_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin);
cudaError_t ring_backward(const tp_desc *d, tp_dtype dtype, const float *grad_out, const void *x, const float *sh,
                          const void *w, const int32_t *src, const int32_t *dst, const int32_t *src_perm,
                          const int32_t *src_row_ptr, int32_t N_src, int32_t N_dst, int64_t E, float *dx, float *dw,
                          float *dsh, void *ws, size_t ws_bytes, int dev, int sms, int smem_optin, int *status,
                          cudaStream_t stream);
cudaError_t mma_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                        const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                        float *out, void *ws, size_t ws_bytes, int dev, int sms, int smem_optin, int *status,
                        cudaStream_t stream);
cudaError_t split_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, int vec_mode,
                          const tp_radial_mlp *mlp, const void *w, const int32_t *src, const int32_t *row_ptr,
                          int32_t N_src, int32_t N_dst, int64_t E, float *out, void *ws, size_t ws_bytes, int dev,
                          int sms, int smem_optin, int *status, cudaStream_t stream);

// ---- process-wide tuning (tp_set_tuning) ----
static std::mutex g_tune_mu;
static tp_tuning g_tune = {};
static uint32_t g_tune_gen = 1;

TuningState tuning_snapshot() {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    return TuningState{g_tune, g_tune_gen};
}
}  // namespace tpc

namespace {

using namespace tpc;

static_assert(sizeof(SegParams) <= 32000, "kernel parameter block too large");

// Device-side status word (TP_DEV_ERR_* bits), one per device the library runs on.
__device__ int g_tp_status;

struct DevInfo {
    int dev = 0;
    int sms = 0;
    int smem_optin = 0;
    int *status = nullptr;
};

std::mutex g_mu;
std::map<int, DevInfo> g_dev;
std::map<std::pair<const void *, int>, int> g_smem_set;  // (kernel, device) -> dynamic smem attribute set

tp_status dev_info(DevInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
        out = it->second;
        return TP_OK;
    }
    DevInfo d;
    d.dev = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TP_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return TP_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tp_status) != cudaSuccess) return TP_ERR_CUDA;
    d.status = static_cast<int *>(p);
    g_dev[dev] = d;
    out = d;
    return TP_OK;
}

tp_status ensure_smem(const void *fn, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(fn, dev);
    auto it = g_smem_set.find(key);
    if (it != g_smem_set.end() && it->second >= bytes) return TP_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return TP_ERR_CUDA;
    g_smem_set[key] = bytes;
    return TP_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Pick edges per chunk, warps per block and the grid for one segment kernel.
tp_status plan_launch(const void *fn, const DevInfo &dev, int head_bytes, int w_bytes, int f_bytes, int sh_floats,
                      int R, bool edge_grad, int n_seg, WarpLayout &L, int &warps, int &grid, int &smem) {
    const int stages = 2;
    const int per_edge = w_bytes + f_bytes + sh_floats * 4;
    int eps = 12288 / per_edge;
    if (eps < 1) eps = 1;
    if (eps > 8) eps = 8;
    const int budget = dev.smem_optin - head_bytes - 1024;
    for (;;) {
        L = make_layout(stages, eps, w_bytes, f_bytes, sh_floats, R, edge_grad);
        if (L.warp_bytes <= budget || eps == 1) break;
        --eps;
    }
    warps = budget / L.warp_bytes;
    if (warps > 8) warps = 8;
    if (warps < 1) return TP_ERR_UNSUPPORTED;
    // no more warps per block than segments need
    if (n_seg < warps) warps = n_seg < 1 ? 1 : n_seg;
    smem = head_bytes + warps * L.warp_bytes;
    tp_status st = ensure_smem(fn, smem);
    if (st != TP_OK) return st;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, warps * 32, smem) != cudaSuccess) return TP_ERR_CUDA;
    if (occ < 1) return TP_ERR_UNSUPPORTED;
    const long long need = (n_seg + warps - 1) / warps;
    const long long cap = (long long)dev.sms * occ;
    grid = (int)(need < cap ? need : cap);
    if (grid < 1) grid = 1;
    return TP_OK;
}

tp_status launch_seg(const void *fn, SegParams &prm, int grid, int warps, int smem, cudaStream_t stream) {
    const TuningState ts = tuning_snapshot();
    prm.wait_ns = ts.t.wait_limit_ns > 0 ? (uint64_t)ts.t.wait_limit_ns : kWaitNs;
    void *args[] = {&prm};
    if (cudaLaunchKernel(fn, dim3(grid), dim3(warps * 32), args, (size_t)smem, stream) != cudaSuccess)
        return TP_ERR_CUDA;
    return TP_OK;
}

}  // namespace

extern "C" tp_status tp_spherical_harmonics(const tp_desc *desc, const float *vec, int64_t E, int32_t normalize,
                                            float *sh, void *stream) {
    if (!desc || E < 0 || (E > 0 && (!vec || !sh))) return TP_ERR_ARG;
    if (E > 0 && (!aligned4(vec) || !aligned4(sh))) return TP_ERR_ALIGN;
    if (sh_launch(vec, E, normalize, desc->tab, sh, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TP_ERR_CUDA;
    return TP_OK;
}

extern "C" tp_status tp_csr_workspace_size(int64_t E, int32_t N, size_t *bytes) {
    if (!bytes || E < 0 || N < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    *bytes = csr_workspace_bytes(E, N);
    return TP_OK;
}

extern "C" tp_status tp_csr_build(const int32_t *keys, int64_t E, int32_t N, int32_t *perm, int32_t *row_ptr,
                                  int32_t *keys_sorted, void *workspace, size_t workspace_bytes, void *stream) {
    if (E < 0 || N < 0 || E >= (int64_t(1) << 31) || !row_ptr) return TP_ERR_ARG;
    if (E > 0 && (!keys || !perm || !workspace)) return TP_ERR_ARG;
    if (E > 0 && N == 0) return TP_ERR_INDEX;
    if (E > 0 && workspace_bytes < csr_workspace_bytes(E, N)) return TP_ERR_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    if (csr_build_launch(keys, E, N, perm, row_ptr, keys_sorted, workspace, dev.status,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TP_ERR_CUDA;
    return TP_OK;
}

extern "C" tp_status tp_csr_build_noalloc(const int32_t *keys, int64_t E, int32_t N, int32_t *perm,
                                          int32_t *row_ptr, int32_t *keys_sorted, void *stream) {
    if (E < 0 || N < 0 || !row_ptr) return TP_ERR_ARG;
    if (E > csr_noalloc_max_edges()) return TP_ERR_CAPACITY;
    if (E > 0 && (!keys || !perm)) return TP_ERR_ARG;
    if (E > 0 && N == 0) return TP_ERR_INDEX;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    void *scratch = nullptr;
    if (csr_noalloc_scratch(&scratch) != cudaSuccess) return TP_ERR_CUDA;
    if (csr_build_launch(keys, E, N, perm, row_ptr, keys_sorted, scratch, dev.status,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TP_ERR_CUDA;
    return TP_OK;
}

extern "C" int64_t tp_csr_build_noalloc_max_edges(void) { return csr_noalloc_max_edges(); }

extern "C" tp_status tp_conv_forward_workspace_size(const tp_desc *desc, tp_dtype dtype, int32_t N_dst, int64_t E,
                                                    size_t *bytes) {
    if (!desc || !bytes || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    const size_t a = split_workspace_bytes(desc, dtype, E, dev.dev, dev.sms, dev.smem_optin);
    const size_t b = mma_workspace_bytes(desc, dtype, E, dev.dev, dev.sms, dev.smem_optin);
    *bytes = a > b ? a : b;
    return TP_OK;
}

namespace {

// Arguments of one forward, after the entry point's own conversions.
struct FwdArgs {
    tp_dtype dtype;
    const void *x;
    const float *sh;  // harmonic rows, or edge vectors when vec_mode != 0
    int vec_mode;     // 0 rows; 1 / 2 vectors (unit / raw harmonics)
    const tp_radial_mlp *mlp;
    const void *w;
    const int32_t *src, *row_ptr;
    int32_t N_src, N_dst;
    int64_t E;
    float *out;
    void *ws;
    size_t ws_bytes;
};

// Checks and dispatch shared by every forward entry point: the tensor-core
// kernel (bfloat16 harmonic rows), the warp-ring kernel, then the generic one
// (harmonic rows only).
tp_status forward_core(const tp_desc *desc, const FwdArgs &a, cudaStream_t stream) {
    if (a.N_src < 0 || a.N_dst < 0 || a.E < 0 || a.E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (a.dtype != TP_F32 && a.dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (a.mlp && (a.dtype != TP_F32 || a.mlp->hidden != 16 || a.vec_mode == 0)) return TP_ERR_UNSUPPORTED;
    if (a.N_dst == 0) return TP_OK;
    if (!a.out || !a.row_ptr) return TP_ERR_ARG;
    if (a.E > 0 && (!a.x || !a.sh || !a.src || (!a.w && !a.mlp))) return TP_ERR_ARG;
    if (a.E > 0 && a.mlp && (!a.mlp->w1 || !a.mlp->b1 || !a.mlp->w2 || !a.mlp->b2)) return TP_ERR_ARG;
    if (a.E > 0 && a.N_src == 0) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    const int esz = a.dtype == TP_F32 ? 4 : 2;
    const int f_bytes = T.dim_x * esz, w_bytes = T.wnum * esz;
    if ((f_bytes & 15) || (w_bytes & 15)) return TP_ERR_ALIGN;
    // weight rows are never read with a radial network: x stands in for the alignment check
    const void *w = a.mlp ? a.x : a.w;
    if (!aligned16(a.out) || (a.E > 0 && (!aligned16(a.x) || !aligned16(w) || !aligned4(a.src) ||
                                          (a.vec_mode ? !aligned16(a.sh) : !aligned4(a.sh)))))
        return TP_ERR_ALIGN;
    if (a.mlp && a.E > 0 &&
        (!aligned4(a.mlp->w1) || !aligned4(a.mlp->b1) || !aligned16(a.mlp->w2) || !aligned16(a.mlp->b2)))
        return TP_ERR_ALIGN;
    if (a.ws && (reinterpret_cast<uintptr_t>(a.ws) & 255u)) return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    if (desc->unsimp) {  // one output block per path: its own kernel (harmonic rows only)
        if (a.vec_mode != 0 || a.mlp) return TP_ERR_UNSUPPORTED;
        const cudaError_t eu = unsimp_forward(desc, a.dtype, a.x, a.sh, a.w, a.src, a.row_ptr, a.N_src, a.N_dst, a.E,
                                              a.out, dev.sms, dev.smem_optin, dev.status, stream);
        if (eu == cudaSuccess) return TP_OK;
        (void)cudaGetLastError();
        return eu == cudaErrorNotSupported ? TP_ERR_UNSUPPORTED : TP_ERR_CUDA;
    }
    cudaError_t e = cudaErrorNotSupported;
    if (a.vec_mode == 0)  // bfloat16 harmonic rows: the tensor-core kernel first
        e = mma_forward(desc, a.dtype, a.x, a.sh, w, a.src, a.row_ptr, a.N_src, a.N_dst, a.E, a.out, a.ws, a.ws_bytes,
                        dev.dev, dev.sms, dev.smem_optin, dev.status, stream);
    if (e == cudaErrorNotSupported)
        e = split_forward(desc, a.dtype, a.x, a.sh, a.vec_mode, a.mlp, w, a.src, a.row_ptr, a.N_src, a.N_dst, a.E,
                          a.out, a.ws, a.ws_bytes, dev.dev, dev.sms, dev.smem_optin, dev.status, stream);
    if (e == cudaSuccess) return TP_OK;
    if (e != cudaErrorNotSupported) return TP_ERR_CUDA;
    (void)cudaGetLastError();
    if (a.vec_mode != 0) return TP_ERR_UNSUPPORTED;  // edge vectors need a compiled kernel and a workspace
    Shape shp;
    if (!pick_shape(desc->lmax_in, desc->lmax_out, shp)) return TP_ERR_UNSUPPORTED;
    const int cpt = pick_cpt(T.mul);
    const void *fn = a.dtype == TP_F32 ? seg_fwd_f32_kernel(shp, cpt) : seg_fwd_bf16_kernel(shp, cpt);
    if (!fn) return TP_ERR_UNSUPPORTED;
    SegParams prm;
    std::memset(&prm, 0, sizeof(prm));
    int warps = 0, grid = 0, smem = 0;
    st = plan_launch(fn, dev, kTablesBytes, w_bytes, f_bytes, T.dim_sh, T.R, false, a.N_dst, prm.lay, warps, grid,
                     smem);
    if (st != TP_OK) return st;
    prm.tab = T;
    prm.feat = a.x;
    prm.sh = a.sh;
    prm.w = a.w;
    prm.gidx = a.src;
    prm.seg_ptr = a.row_ptr;
    prm.out = a.out;
    prm.status = dev.status;
    prm.n_seg = a.N_dst;
    prm.n_gather = a.N_src;
    prm.n_edges = a.E;
    return launch_seg(fn, prm, grid, warps, smem, stream);
}

}  // namespace

extern "C" tp_status tp_conv_forward(const tp_desc *desc, tp_dtype dtype, const void *x, const float *sh, const void *w,
                                     const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst,
                                     int64_t E, float *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc) return TP_ERR_ARG;
    if (desc->layout != TP_IR_MUL) return TP_ERR_UNSUPPORTED;
    const FwdArgs a{dtype, x, sh, 0, nullptr, w, src, row_ptr, N_src, N_dst, E, out, workspace, workspace_bytes};
    return forward_core(desc, a, static_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_conv_forward_vec(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const void *w, const int32_t *src, const int32_t *row_ptr,
                                         int32_t N_src, int32_t N_dst, int64_t E, float *out, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    if (!desc) return TP_ERR_ARG;
    if (desc->layout != TP_IR_MUL) return TP_ERR_UNSUPPORTED;
    const FwdArgs a{dtype, x, vec, normalize ? 1 : 2, nullptr, w, src, row_ptr, N_src, N_dst, E, out, workspace,
                    workspace_bytes};
    return forward_core(desc, a, static_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_conv_forward_mlp(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const tp_radial_mlp *mlp, const int32_t *src,
                                         const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E, float *out,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc || !mlp) return TP_ERR_ARG;
    if (desc->layout != TP_IR_MUL) return TP_ERR_UNSUPPORTED;
    const FwdArgs a{dtype, x, vec, normalize ? 1 : 2, mlp, nullptr, src, row_ptr, N_src, N_dst, E, out, workspace,
                    workspace_bytes};
    return forward_core(desc, a, static_cast<cudaStream_t>(stream));
}

// ---- tp_conv_forward_ex: index width, layout and reduction around the core ----

namespace {

size_t al256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of tp_conv_forward_ex: the core forward's, then (as needed) int32
// copies of src and row_ptr, an ir_mul copy of x and an ir_mul out.
struct ExLayout {
    size_t core, src32, rp32, x_ir, out_ir, total;
};

tp_status ex_layout(const tp_desc *desc, const tp_forward_args *a, ExLayout &L) {
    if (!a || a->N_src < 0 || a->N_dst < 0 || a->E < 0 || a->E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (a->dtype != TP_F32 && a->dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (a->index_bits != 32 && a->index_bits != 64) return TP_ERR_ARG;
    if (a->reduce != TP_REDUCE_SUM && a->reduce != TP_REDUCE_MEAN) return TP_ERR_ARG;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    const size_t c1 = split_workspace_bytes(desc, a->dtype, a->E, dev.dev, dev.sms, dev.smem_optin);
    const size_t c2 = a->vec ? 0 : mma_workspace_bytes(desc, a->dtype, a->E, dev.dev, dev.sms, dev.smem_optin);
    const Tables &T = desc->tab;
    const size_t esz = a->dtype == TP_F32 ? 4 : 2;
    const bool i64 = a->index_bits == 64, mi = desc->layout == TP_MUL_IR;
    L.core = al256(c1 > c2 ? c1 : c2);
    L.src32 = L.core;
    L.rp32 = L.src32 + (i64 ? al256((size_t)a->E * 4) : 0);
    L.x_ir = L.rp32 + (i64 ? al256(((size_t)a->N_dst + 1) * 4) : 0);
    L.out_ir = L.x_ir + (mi ? al256((size_t)a->N_src * T.dim_x * esz) : 0);
    L.total = L.out_ir + (mi ? al256((size_t)a->N_dst * T.dim_out * 4) : 0);
    return TP_OK;
}

}  // namespace

extern "C" tp_status tp_conv_forward_ex_workspace_size(const tp_desc *desc, const tp_forward_args *args,
                                                       size_t *bytes) {
    if (!desc || !bytes) return TP_ERR_ARG;
    ExLayout L;
    const tp_status st = ex_layout(desc, args, L);
    if (st != TP_OK) return st;
    *bytes = L.total;
    return TP_OK;
}

extern "C" tp_status tp_conv_forward_ex(const tp_desc *desc, const tp_forward_args *a, void *stream) {
    if (!desc || !a) return TP_ERR_ARG;
    ExLayout L;
    tp_status st = ex_layout(desc, a, L);
    if (st != TP_OK) return st;
    if (a->N_dst == 0) return TP_OK;
    if (!a->workspace || a->workspace_bytes < L.total) return TP_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return TP_ERR_ALIGN;
    if (!a->out || !a->row_ptr || (a->E > 0 && (!a->x || !a->src))) return TP_ERR_ARG;
    if (a->sh && a->vec) return TP_ERR_ARG;  // harmonic rows or edge vectors, not both
    if (a->mlp && !a->vec) return TP_ERR_UNSUPPORTED;
    if (desc->unsimp && a->reduce != TP_REDUCE_SUM) return TP_ERR_UNSUPPORTED;
    DevInfo dev;
    st = dev_info(dev);
    if (st != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(a->workspace);
    const Tables &T = desc->tab;
    const int esz = a->dtype == TP_F32 ? 4 : 2;
    const int32_t *src = static_cast<const int32_t *>(a->src), *rp = static_cast<const int32_t *>(a->row_ptr);
    if (a->index_bits == 64) {  // int32 copies (out-of-range values become invalid indices the kernels flag)
        if (indices_to_i32(static_cast<const int64_t *>(a->src), a->E, reinterpret_cast<int32_t *>(ws + L.src32), s) !=
                cudaSuccess ||
            indices_to_i32(static_cast<const int64_t *>(a->row_ptr), (int64_t)a->N_dst + 1,
                           reinterpret_cast<int32_t *>(ws + L.rp32), s) != cudaSuccess)
            return TP_ERR_CUDA;
        src = reinterpret_cast<const int32_t *>(ws + L.src32);
        rp = reinterpret_cast<const int32_t *>(ws + L.rp32);
    }
    const void *x = a->x;
    float *out = a->out;
    if (desc->layout == TP_MUL_IR) {
        if (a->N_src > 0 && a->E > 0 &&
            transpose_rows(desc, 0, TP_MUL_IR, a->x, ws + L.x_ir, a->N_src, esz, s) != cudaSuccess)
            return TP_ERR_CUDA;
        x = ws + L.x_ir;
        out = reinterpret_cast<float *>(ws + L.out_ir);
    }
    const FwdArgs f{a->dtype, x, a->vec ? a->vec : a->sh, a->vec ? (a->normalize ? 1 : 2) : 0, a->mlp, a->w, src, rp,
                    a->N_src, a->N_dst, a->E, out, a->workspace, L.core};
    st = forward_core(desc, f, s);
    if (st != TP_OK) return st;
    if (a->reduce == TP_REDUCE_MEAN && scale_rows_by_inverse_degree(out, rp, a->N_dst, T.dim_out, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (desc->layout == TP_MUL_IR && transpose_rows(desc, 1, TP_IR_MUL, out, a->out, a->N_dst, 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    return TP_OK;
}

extern "C" tp_status tp_transpose_layout(const tp_desc *desc, int32_t which, tp_layout from, const void *src,
                                         void *dst, int64_t rows, int32_t elem_bytes, void *stream) {
    if (!desc || (which != 0 && which != 1) || (from != TP_IR_MUL && from != TP_MUL_IR) || rows < 0 ||
        (elem_bytes != 2 && elem_bytes != 4))
        return TP_ERR_ARG;
    if (rows == 0) return TP_OK;
    if (!src || !dst || src == dst) return TP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & (uintptr_t)(elem_bytes - 1))
        return TP_ERR_ALIGN;
    return transpose_rows(desc, which, from, src, dst, rows, elem_bytes, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TP_OK
               : TP_ERR_CUDA;
}

extern "C" tp_status tp_conv_backward_workspace_size(const tp_desc *desc, tp_dtype dtype, int32_t N_src, int64_t E,
                                                     size_t *bytes) {
    if (!desc || !bytes || N_src < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    *bytes = ring_bwd_workspace_bytes(desc, dtype, E, dev.dev, dev.sms, dev.smem_optin);
    return TP_OK;
}

extern "C" tp_status tp_conv_backward(const tp_desc *desc, tp_dtype dtype, const float *grad_out, const void *x,
                                      const float *sh, const void *w, const int32_t *src, const int32_t *dst,
                                      const int32_t *row_ptr, const int32_t *src_perm, const int32_t *src_row_ptr,
                                      int32_t N_src, int32_t N_dst, int64_t E, float *dx, float *dw, float *dsh,
                                      void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc || N_src < 0 || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (desc->layout != TP_IR_MUL || desc->unsimp) return TP_ERR_UNSUPPORTED;
    if ((N_src > 0 && (!dx || !src_row_ptr)) || (N_dst > 0 && !row_ptr)) return TP_ERR_ARG;
    if (E > 0 && (!grad_out || !x || !sh || !w || !src || !dst || !src_perm || !dw || !dsh)) return TP_ERR_ARG;
    if (E > 0 && (N_src == 0 || N_dst == 0)) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    const int esz = dtype == TP_F32 ? 4 : 2;
    if (((T.dim_x * esz) & 15) || ((T.wnum * esz) & 15) || ((T.dim_out * 4) & 15) || ((T.wnum * 4) & 15))
        return TP_ERR_ALIGN;
    if ((dx && !aligned16(dx)) ||
        (E > 0 && (!aligned16(grad_out) || !aligned16(x) || !aligned16(w) || !aligned16(dw) || !aligned4(sh) ||
                   !aligned4(dsh))) ||
        (workspace && !aligned16(workspace)))
        return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N_src > 0) {
        const cudaError_t e = ring_backward(desc, dtype, grad_out, x, sh, w, src, dst, src_perm, src_row_ptr, N_src,
                                            N_dst, E, dx, dw, dsh, workspace, workspace_bytes, dev.dev, dev.sms,
                                            dev.smem_optin, dev.status, s);
        if (e == cudaSuccess) return TP_OK;
        if (e != cudaErrorNotSupported) {
            (void)cudaGetLastError();
            return TP_ERR_CUDA;
        }
    }
    // the generic two-kernel backward: float32, any descriptor the seg kernels cover
    if (dtype != TP_F32) return TP_ERR_UNSUPPORTED;
    Shape shp;
    if (!pick_shape(desc->lmax_in, desc->lmax_out, shp)) return TP_ERR_UNSUPPORTED;
    const int cpt = pick_cpt(T.mul);
    if (E > 0 && N_dst > 0) {  // dw, dsh: warp per destination
        const void *fn = seg_bwde_f32_kernel(shp, cpt);
        if (!fn) return TP_ERR_UNSUPPORTED;
        SegParams prm;
        std::memset(&prm, 0, sizeof(prm));
        int warps = 0, grid = 0, smem = 0;
        st = plan_launch(fn, dev, kTablesBytes + kTrTablesBytes, T.wnum * 4, T.dim_x * 4, T.dim_sh, T.R, true, N_dst,
                         prm.lay, warps, grid, smem);
        if (st != TP_OK) return st;
        prm.tab = T;
        prm.feat = x;
        prm.sh = sh;
        prm.w = w;
        prm.gidx = src;
        prm.seg_ptr = row_ptr;
        prm.g = grad_out;
        prm.dw = dw;
        prm.dsh = dsh;
        prm.status = dev.status;
        prm.n_seg = N_dst;
        prm.n_gather = N_src;
        prm.n_edges = E;
        st = launch_seg(fn, prm, grid, warps, smem, s);
        if (st != TP_OK) return st;
    }
    if (N_src > 0) {  // dx: warp per source
        const void *fn = seg_bwdx_f32_kernel(shp, cpt);
        if (!fn) return TP_ERR_UNSUPPORTED;
        SegParams prm;
        std::memset(&prm, 0, sizeof(prm));
        int warps = 0, grid = 0, smem = 0;
        st = plan_launch(fn, dev, kTablesBytes, T.wnum * 4, T.dim_out * 4, T.dim_sh, T.R, false, N_src, prm.lay, warps,
                         grid, smem);
        if (st != TP_OK) return st;
        prm.tab = T;
        prm.feat = grad_out;
        prm.sh = sh;
        prm.w = w;
        prm.gidx = dst;
        prm.seg_ptr = src_row_ptr;
        prm.slot_edge = src_perm;
        prm.out = dx;
        prm.status = dev.status;
        prm.n_seg = N_src;
        prm.n_gather = N_dst;
        prm.n_edges = E;
        st = launch_seg(fn, prm, grid, warps, smem, s);
        if (st != TP_OK) return st;
    }
    return TP_OK;
}

extern "C" tp_status tp_set_tuning(const tp_tuning *t) {
    tp_tuning v = {};
    if (t) {
        v = *t;
        const bool ok = v.ring_stage_bytes >= 0 && (v.ring_stages == 0 || (v.ring_stages >= 2 && v.ring_stages <= 8)) &&
                        (v.ring_warps == 0 || (v.ring_warps >= 1 && v.ring_warps <= kRingMaxWarps)) &&
                        (v.ring_rounds == 0 || (v.ring_rounds >= 1 && v.ring_rounds <= kRingMaxPiecesPerWarp)) &&
                        v.ring_pack >= 0 && v.ring_pack <= 2 && (v.disable_split == 0 || v.disable_split == 1) &&
                        v.wait_limit_ns >= 0 && (v.disable_mma == 0 || v.disable_mma == 1) &&
                        (v.mma_stages == 0 || (v.mma_stages >= 3 && v.mma_stages <= 8)) &&
                        v.bwd_stage_bytes >= 0 && (v.bwd_stages == 0 || (v.bwd_stages >= 2 && v.bwd_stages <= 8)) &&
                        (v.bwd_warps == 0 || (v.bwd_warps >= 1 && v.bwd_warps <= kRingMaxWarps)) &&
                        (v.disable_ring_bwd == 0 || v.disable_ring_bwd == 1) &&
                        (v.disable_symc_jit == 0 || v.disable_symc_jit == 1);
        if (!ok) return TP_ERR_ARG;
    }
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tune = v;
    ++g_tune_gen;
    return TP_OK;
}

extern "C" tp_status tp_get_tuning(tp_tuning *t) {
    if (!t) return TP_ERR_ARG;
    *t = tuning_snapshot().t;
    return TP_OK;
}

extern "C" tp_status tp_symmetric_contraction(const tp_symc *symc, const float *x, const float *weights,
                                              const int32_t *element, int32_t N, int32_t num_elements, float *out,
                                              void *stream) {
    if (!symc || N < 0 || num_elements < 1) return TP_ERR_ARG;
    if (N == 0) return TP_OK;
    if (!x || !weights || !element || !out) return TP_ERR_ARG;
    if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(weights) & 7u) || !aligned4(element))
        return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorNotSupported;
    if (!tuning_snapshot().t.disable_symc_jit)  // the kernel specialised for this descriptor
        e = symc_jit_launch(symc, x, weights, element, N, num_elements, out, dev.dev, dev.sms, dev.status, s);
    if (e == cudaErrorNotSupported)  // the table kernel
        e = symc_launch(symc, x, weights, element, N, num_elements, out, dev.sms, dev.smem_optin, dev.status, s);
    if (e == cudaSuccess) return TP_OK;
    (void)cudaGetLastError();
    return e == cudaErrorNotSupported ? TP_ERR_UNSUPPORTED : TP_ERR_CUDA;
}

extern "C" tp_status tp_device_status(int32_t *flags, int32_t reset, void *stream) {
    if (!flags) return TP_ERR_ARG;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, dev.status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return TP_ERR_CUDA;
    if (reset && cudaMemsetAsync(dev.status, 0, sizeof(int), s) != cudaSuccess) return TP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TP_ERR_CUDA;
    *flags = v;
    return TP_OK;
}

extern "C" const char *tp_status_string(tp_status s) {
    switch (s) {
        case TP_OK: return "ok";
        case TP_ERR_PARSE: return "irreps string cannot be parsed";
        case TP_ERR_UNSUPPORTED: return "configuration not supported by the kernels";
        case TP_ERR_INDEX: return "index out of range";
        case TP_ERR_ALIGN: return "pointer or row size not 16-byte aligned";
        case TP_ERR_CUDA: return "CUDA runtime error";
        case TP_ERR_ARG: return "invalid argument";
        case TP_ERR_TIMEOUT: return "device pipeline wait timed out";
        case TP_ERR_CAPACITY: return "size exceeds the fixed scratch capacity of this entry point";
    }
    return "unknown status";
}

extern "C" int32_t tp_abi_version(void) { return TPCONV_ABI_VERSION; }
