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
size_t mma_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin);
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

extern "C" tp_status tp_conv_forward(const tp_desc *desc, tp_dtype dtype, const void *x, const float *sh, const void *w,
                                     const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst,
                                     int64_t E, float *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc || N_src < 0 || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (N_dst == 0) return TP_OK;
    if (!out || !row_ptr) return TP_ERR_ARG;
    if (E > 0 && (!x || !sh || !w || !src)) return TP_ERR_ARG;
    if (E > 0 && N_src == 0) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    const int esz = dtype == TP_F32 ? 4 : 2;
    const int f_bytes = T.dim_x * esz, w_bytes = T.wnum * esz;
    if ((f_bytes & 15) || (w_bytes & 15)) return TP_ERR_ALIGN;
    if (!aligned16(out) || (E > 0 && (!aligned16(x) || !aligned16(w) || !aligned4(sh) || !aligned4(src))))
        return TP_ERR_ALIGN;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TP_ERR_ALIGN;
    {
        DevInfo dev;
        tp_status st = dev_info(dev);
        if (st != TP_OK) return st;
        // bfloat16 inputs: the tensor-core kernel first
        cudaError_t e = mma_forward(desc, dtype, x, sh, w, src, row_ptr, N_src, N_dst, E, out, workspace,
                                    workspace_bytes, dev.dev, dev.sms, dev.smem_optin, dev.status,
                                    static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) return TP_OK;
        if (e != cudaErrorNotSupported) return TP_ERR_CUDA;
        e = split_forward(desc, dtype, x, sh, 0, nullptr, w, src, row_ptr, N_src, N_dst, E, out, workspace,
                                           workspace_bytes, dev.dev, dev.sms, dev.smem_optin, dev.status,
                                           static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) return TP_OK;
        if (e != cudaErrorNotSupported) return TP_ERR_CUDA;
        (void)cudaGetLastError();
    }
    Shape shp;
    if (!pick_shape(desc->lmax_in, desc->lmax_out, shp)) return TP_ERR_UNSUPPORTED;
    const int cpt = pick_cpt(T.mul);
    const void *fn = dtype == TP_F32 ? seg_fwd_f32_kernel(shp, cpt) : seg_fwd_bf16_kernel(shp, cpt);
    if (!fn) return TP_ERR_UNSUPPORTED;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    SegParams prm;
    std::memset(&prm, 0, sizeof(prm));
    int warps = 0, grid = 0, smem = 0;
    st = plan_launch(fn, dev, kTablesBytes, w_bytes, f_bytes, T.dim_sh, T.R, false, N_dst, prm.lay, warps, grid, smem);
    if (st != TP_OK) return st;
    prm.tab = T;
    prm.feat = x;
    prm.sh = sh;
    prm.w = w;
    prm.gidx = src;
    prm.seg_ptr = row_ptr;
    prm.out = out;
    prm.status = dev.status;
    prm.n_seg = N_dst;
    prm.n_gather = N_src;
    prm.n_edges = E;
    return launch_seg(fn, prm, grid, warps, smem, static_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_conv_forward_vec(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const void *w, const int32_t *src, const int32_t *row_ptr,
                                         int32_t N_src, int32_t N_dst, int64_t E, float *out, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    if (!desc || N_src < 0 || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (N_dst == 0) return TP_OK;
    if (!out || !row_ptr) return TP_ERR_ARG;
    if (E > 0 && (!x || !vec || !w || !src)) return TP_ERR_ARG;
    if (E > 0 && N_src == 0) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    const int esz = dtype == TP_F32 ? 4 : 2;
    if (((T.dim_x * esz) & 15) || ((T.wnum * esz) & 15)) return TP_ERR_ALIGN;
    if (!aligned16(out) || (E > 0 && (!aligned16(x) || !aligned16(w) || !aligned16(vec) || !aligned4(src))))
        return TP_ERR_ALIGN;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    const cudaError_t e = split_forward(desc, dtype, x, vec, normalize ? 1 : 2, nullptr, w, src, row_ptr, N_src, N_dst, E, out,
                                       workspace, workspace_bytes, dev.dev, dev.sms, dev.smem_optin, dev.status,
                                       static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return TP_OK;
    (void)cudaGetLastError();
    return e == cudaErrorNotSupported ? TP_ERR_UNSUPPORTED : TP_ERR_CUDA;
}

extern "C" tp_status tp_conv_forward_mlp(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const tp_radial_mlp *mlp, const int32_t *src,
                                         const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E, float *out,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc || !mlp || N_src < 0 || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if (dtype != TP_F32 && dtype != TP_BF16_IN_F32_OUT) return TP_ERR_ARG;
    if (dtype != TP_F32 || mlp->hidden != 16) return TP_ERR_UNSUPPORTED;
    if (N_dst == 0) return TP_OK;
    if (!out || !row_ptr) return TP_ERR_ARG;
    if (E > 0 && (!x || !vec || !src || !mlp->w1 || !mlp->b1 || !mlp->w2 || !mlp->b2)) return TP_ERR_ARG;
    if (E > 0 && N_src == 0) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    if ((T.dim_x * 4) & 15) return TP_ERR_ALIGN;
    if (!aligned16(out) || (E > 0 && (!aligned16(x) || !aligned16(vec) || !aligned4(src) || !aligned4(mlp->w1) ||
                                      !aligned4(mlp->b1) || !aligned4(mlp->w2) || !aligned4(mlp->b2))))
        return TP_ERR_ALIGN;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TP_ERR_ALIGN;
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    // w is never read in this mode; the weight-row pointer only has to qualify the alignment check
    const cudaError_t e = split_forward(desc, dtype, x, vec, normalize ? 1 : 2, mlp, x, src, row_ptr, N_src, N_dst, E,
                                       out, workspace, workspace_bytes, dev.dev, dev.sms, dev.smem_optin, dev.status,
                                       static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return TP_OK;
    (void)cudaGetLastError();
    return e == cudaErrorNotSupported ? TP_ERR_UNSUPPORTED : TP_ERR_CUDA;
}

extern "C" tp_status tp_conv_backward(const tp_desc *desc, const float *grad_out, const float *x, const float *sh,
                                      const float *w, const int32_t *src, const int32_t *dst, const int32_t *row_ptr,
                                      const int32_t *src_perm, const int32_t *src_row_ptr, int32_t N_src,
                                      int32_t N_dst, int64_t E, float *dx, float *dw, float *dsh, void *stream) {
    if (!desc || N_src < 0 || N_dst < 0 || E < 0 || E >= (int64_t(1) << 31)) return TP_ERR_ARG;
    if ((N_src > 0 && (!dx || !src_row_ptr)) || (N_dst > 0 && !row_ptr)) return TP_ERR_ARG;
    if (E > 0 && (!grad_out || !x || !sh || !w || !src || !dst || !src_perm || !dw || !dsh)) return TP_ERR_ARG;
    if (E > 0 && (N_src == 0 || N_dst == 0)) return TP_ERR_INDEX;
    const Tables &T = desc->tab;
    if (((T.dim_x * 4) & 15) || ((T.wnum * 4) & 15) || ((T.dim_out * 4) & 15)) return TP_ERR_ALIGN;
    if ((dx && !aligned16(dx)) ||
        (E > 0 && (!aligned16(grad_out) || !aligned16(x) || !aligned16(w) || !aligned16(dw) || !aligned4(sh) ||
                   !aligned4(dsh))))
        return TP_ERR_ALIGN;
    Shape shp;
    if (!pick_shape(desc->lmax_in, desc->lmax_out, shp)) return TP_ERR_UNSUPPORTED;
    const int cpt = pick_cpt(T.mul);
    DevInfo dev;
    tp_status st = dev_info(dev);
    if (st != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
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
                        (v.mma_stages == 0 || (v.mma_stages >= 3 && v.mma_stages <= 8));
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
