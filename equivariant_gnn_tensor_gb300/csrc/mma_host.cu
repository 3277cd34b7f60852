// Host side of the tensor-core forward (mma_fwd.cuh): eligibility, the Mbig
// entry table, the 2-D tensor map of x, shared-memory layout, launch of the
// kernel and of the partial-row merge.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>

#include "mma_fwd.cuh"
#include "tuning.h"

namespace tpc {

namespace {

using Shape333 = MmaShape<3, 3, 3>;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once.
EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The launch-independent part: parameters with the layout and the Mbig
// entries, occupancy, kernel.
struct MmaPlan {
    const void *fn = nullptr;
    MmaParams prm{};
    int smem = 0, occ = 0;
};

bool mma_plan(const tp_desc *d, int smem_optin, const tp_tuning &tu, MmaPlan &pl) {
    const ProgramPlan &TP = d->prog;
    const Tables &T = d->tab;
    if (!TP.valid || T.mul != kMmaMul) return false;
    const ProgShape shp = kProgShapes[TP.shape];
    if (shp.li != 3 || shp.lsh != 3 || shp.lo != 3) return false;
    constexpr Program P = Shape333::P;
    // natural layout: block l at l*l*mul, paths in program order
    if (T.dim_x != 16 * kMmaMul || T.dim_out != 16 * kMmaMul || T.dim_sh != 16 || T.wnum != P.n * kMmaMul ||
        TP.R != P.R)
        return false;
    for (int l = 0; l <= 3; ++l)
        if (T.x_off[l] != l * l * kMmaMul || T.o_off[l] != l * l * kMmaMul) return false;
    for (int t = 0; t < P.n; ++t)
        if (TP.wofs[t] != t * kMmaMul) return false;
    MmaParams &g = pl.prm;
    std::memset(&g, 0, sizeof(g));
    // Mbig entries of every path: row la^2 + i, column col0(t) + k of the
    // K-major B operand (8 x 16-byte core matrices: K step 128 B, N step 256 B)
    int n = 0;
    for (int t = 0; t < P.n; ++t) {
        const int la = P.p[t].la, c0 = Shape333::col0(t);
        for (int q = 0; q < P.nz[t]; ++q) {
            const int r = P.moff[t] + q;
            const int krow = la * la + (P.ik[t][q] >> 3), col = c0 + (P.ik[t][q] & 7);
            if (n >= kMmaMaxEnt) return false;
            g.ent_off[n] = (uint16_t)((col / 8) * 256 + (krow / 8) * 128 + (col % 8) * 16 + (krow % 8) * 2);
            const uint32_t j0 = TP.ej[r] & 0xffffu, j1 = TP.ej[r] >> 16;
            if (j0 > 15 || j1 > 15) return false;
            g.ent_j[n] = (uint8_t)(j0 | (j1 << 4));
            g.ent_c[n][0] = TP.ec[r][0];
            g.ent_c[n][1] = TP.ec[r][1];
            ++n;
        }
    }
    g.n_ent = n;
    // stages; at least enough shared memory that no third CTA fits on an SM
    // (two CTAs use all 512 tensor-memory columns)
    const int S = tu.mma_stages ? tu.mma_stages : 6;
    const int MB = Shape333::MB_BYTES, WB = Shape333::WB_BYTES, SHB = Shape333::SH_BYTES;
    int off = 0;
    g.S = S;
    g.z0_off = off;
    off += 2048;
    g.x_off = off;
    off += S * 4096;
    g.z1_off = off;
    off += 2048;
    g.m_off = off;
    off += 4 * kMmaMStages * MB;
    g.w_off = off;
    off += 2 * S * WB;
    g.sh_off = off;
    off += 2 * S * SHB;
    g.bar_off = (off + 15) / 16 * 16;
    off = g.bar_off + (2 * S + 2 * kMmaMStages + 4) * 8 + 16;
    int smem = off + 1024;  // room to align the base to 1024 bytes
    if (smem > smem_optin) return false;
    pl.fn = reinterpret_cast<const void *>(&mma_fwd_kernel<3, 3, 3>);
    if (cudaFuncSetAttribute(pl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) != cudaSuccess)
        return false;
    // two CTAs per SM share its 512 tensor-memory columns: never three, so the
    // request is padded to more than a third of the SM's shared memory
    int per_sm = 0, dev = 0, reserved = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return false;
    if (smem < per_sm / 3 + 1024) smem = per_sm / 3 + 1024;
    if (smem > smem_optin) return false;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pl.fn) != cudaSuccess) return false;
    const int occ_smem = per_sm / (smem + reserved);
    const int occ_regs = 65536 / (fa.numRegs * kMmaThreads);
    int occ = occ_smem < occ_regs ? occ_smem : occ_regs;
    if (occ > 2) occ = 2;
    if (occ < 1) return false;
    g.smem_bytes = smem;
    pl.smem = smem;
    pl.occ = occ;
    return true;
}

struct PlanKey {
    uint64_t uid;
    int dev;
    uint32_t gen;
    bool operator<(const PlanKey &o) const { return std::tie(uid, dev, gen) < std::tie(o.uid, o.dev, o.gen); }
};
std::mutex g_mu;
std::map<PlanKey, std::unique_ptr<MmaPlan>> g_plans;  // nullptr: not eligible

const MmaPlan *cached_plan(const tp_desc *d, int dev, int smem_optin, const TuningState &ts) {
    const PlanKey key{d->uid, dev, ts.gen};
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) return it->second.get();
    std::unique_ptr<MmaPlan> pl(new MmaPlan());
    if (!mma_plan(d, smem_optin, ts.t, *pl)) pl.reset();
    const MmaPlan *p = pl.get();
    g_plans[key] = std::move(pl);
    return p;
}

size_t carry_bytes(int pieces, int dim_out) {
    const size_t a = (size_t)2 * pieces * dim_out * sizeof(float);
    return (a + 255) / 256 * 256 + (size_t)2 * pieces * sizeof(int32_t);
}

// CTAs for E edges: two per SM, but at least ~32 edges per CTA (a CTA walks
// its edge pairs one stage after another; on a small graph more CTAs keep more
// of them in flight).
int mma_ctas(const MmaPlan &pl, int64_t E, int sms) {
    long long c = (long long)sms * pl.occ;
    const long long by_edges = (E + 31) / 32;
    if (c > by_edges) c = by_edges;
    return c < 1 ? 1 : (int)c;
}

}  // namespace

void mma_cache_forget(uint64_t uid) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto it = g_plans.begin(); it != g_plans.end();) it = it->first.uid == uid ? g_plans.erase(it) : std::next(it);
}

// Workspace of the tensor-core forward (0: not eligible).
size_t mma_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin) {
    const TuningState ts = tuning_snapshot();
    if (dtype != TP_BF16_IN_F32_OUT || ts.t.disable_mma || ts.t.disable_split || E <= 0 || E >= (int64_t)1 << 31)
        return 0;
    const MmaPlan *pl = cached_plan(d, dev, smem_optin, ts);
    if (!pl || !encode_fn()) return 0;
    return carry_bytes(2 * mma_ctas(*pl, E, sms), d->tab.dim_out);
}

// Launches the tensor-core forward (+ partial merge). cudaErrorNotSupported
// when the call does not qualify (the caller then tries the other kernels).
cudaError_t mma_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                        const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                        float *out, void *ws, size_t ws_bytes, int dev, int sms, int smem_optin, int *status,
                        cudaStream_t stream) {
    const TuningState ts = tuning_snapshot();
    if (dtype != TP_BF16_IN_F32_OUT || ts.t.disable_mma || ts.t.disable_split || !ws || E <= 0 ||
        E >= (int64_t)1 << 31 || N_src <= 0 || (int64_t)N_src * 16 >= ((int64_t)1 << 31))
        return cudaErrorNotSupported;
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                         reinterpret_cast<uintptr_t>(sh);
    if ((al & 15u) != 0) return cudaErrorNotSupported;
    const MmaPlan *pl = cached_plan(d, dev, smem_optin, ts);
    EncodeTiledFn enc = encode_fn();
    if (!pl || !enc) return cudaErrorNotSupported;
    const int n_ctas = mma_ctas(*pl, E, sms);
    const int n_pieces = 2 * n_ctas;
    const int dim_out = d->tab.dim_out;
    if (carry_bytes(n_pieces, dim_out) > ws_bytes) return cudaErrorNotSupported;
    // x as rows of 64 bf16 (one 16-row block per node), read in 16 x 64 boxes
    // with the 128-byte swizzle of the MMA's MN-major operand layout
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)kMmaMul, (cuuint64_t)N_src * 16};
    const cuuint64_t gstride[1] = {(cuuint64_t)kMmaMul * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kMmaMul, 16};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    static_assert(sizeof(MmaParams) + sizeof(CUtensorMap) < 32000, "kernel parameter block too large");
    MmaParams prm = pl->prm;
    prm.w = w;
    prm.sh = sh;
    prm.src = src;
    prm.row_ptr = row_ptr;
    prm.out = out;
    prm.carry = static_cast<float *>(ws);
    const size_t cb = ((size_t)2 * n_pieces * dim_out * sizeof(float) + 255) / 256 * 256;
    prm.carry_dst = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + cb);
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.n_pieces = n_pieces;
    prm.E = E;
    prm.wait_ns = ts.t.wait_limit_ns > 0 ? (uint64_t)ts.t.wait_limit_ns : kWaitNs;
    void *args[] = {&tmap, &prm};
    cudaError_t e = cudaLaunchKernel(pl->fn, dim3(n_ctas), dim3(kMmaThreads), args, (size_t)pl->smem, stream);
    if (e != cudaSuccess) return e;
    const int wpb = 8;
    carry_fixup_kernel<<<(n_pieces + wpb - 1) / wpb, 32 * wpb, 0, stream>>>(prm.carry, prm.carry_dst, n_pieces,
                                                                            dim_out, N_dst, out);
    return cudaGetLastError();
}

}  // namespace tpc
