// Host side of the program-specialised backward (ring_bwd.cuh): launch plan
// (kernel, per-warp shared-memory ring, M recipe and the harmonic-gradient
// coefficients), its cache, the workspace for partial dx rows of sources cut
// by piece boundaries, and the launch with the partial merge.
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>

#include "ring_bwd.cuh"
#include "tuning.h"

namespace tpc {

const void *ring_bwd_kernel_f32(int shape, int cpt);
const void *ring_bwd_kernel_bf16(int shape, int cpt);

namespace {

struct BwdLaunch {
    const void *fn = nullptr;
    RingBwdParams geo{};  // layout fields and tables only
    int wpb = 0, smem = 0, occ = 0;
};

size_t bwd_carry_bytes(int pieces, int dim_x) {
    const size_t a = (size_t)2 * pieces * dim_x * sizeof(float);
    return (a + 255) / 256 * 256 + (size_t)2 * pieces * sizeof(int32_t);
}

// The descriptor must be in the natural layout of a compiled program (as for
// the forward ring kernel), and every Clebsch-Gordan term of every M entry
// must sit on one of the entry's compile-time harmonic components.
bool bwd_plan(const tp_desc *d, tp_dtype dtype, int smem_optin, const tp_tuning &tu, BwdLaunch &bl) {
    const ProgramPlan &TP = d->prog;
    if (!TP.valid || tu.disable_ring_bwd) return false;
    const Tables &T = d->tab;
    const int mul = T.mul;
    if (mul % 32 != 0) return false;
    const int cpt = mul / 32;
    if (cpt != 1 && cpt != 2 && cpt != 4) return false;
    const ProgShape shp = kProgShapes[TP.shape];
    const Program prog = make_natural_program(shp.li, shp.lsh, shp.lo);
    if (T.dim_x != (shp.li + 1) * (shp.li + 1) * mul || T.dim_out != (shp.lo + 1) * (shp.lo + 1) * mul ||
        T.dim_sh != (shp.lsh + 1) * (shp.lsh + 1) || T.wnum != prog.n * mul || TP.R != prog.R)
        return false;
    for (int l = 0; l <= shp.li; ++l)
        if (T.x_off[l] != l * l * mul) return false;
    for (int l = 0; l <= shp.lo; ++l)
        if (T.o_off[l] != l * l * mul) return false;
    for (int t = 0; t < prog.n; ++t)
        if (TP.wofs[t] != t * mul) return false;
    bl.fn = dtype == TP_F32 ? ring_bwd_kernel_f32(TP.shape, cpt) : ring_bwd_kernel_bf16(TP.shape, cpt);
    if (!bl.fn) return false;
    RingBwdParams &g = bl.geo;
    std::memset(&g, 0, sizeof(g));
    std::memcpy(g.ej, TP.ej, sizeof(uint32_t) * TP.R);
    std::memcpy(g.ec, TP.ec, sizeof(float) * 2 * TP.R);
    // coefficients per compile-time component slot: M entry r = sum_slot cc[r][slot] * sh[j(slot)]
    for (int t = 0; t < prog.n; ++t) {
        const ProgPath pp = prog.p[t];
        for (int q = 0; q < prog.nz[t]; ++q) {
            const int r = prog.moff[t] + q;
            const int i = prog.ik[t][q] >> 3, k = prog.ik[t][q] & 7;
            for (int term = 0; term < 2; ++term) {
                const float c = TP.ec[r][term];
                if (c == 0.f) continue;
                const int jg = (int)(term == 0 ? (TP.ej[r] & 0xffffu) : (TP.ej[r] >> 16));
                int slot = -1;
                for (int sl = 0; sl < 2; ++sl) {
                    const int j = m_entry_j(pp.la, pp.lb, pp.lc, i, k, sl);
                    if (j >= 0 && pp.lb * pp.lb + j == jg) slot = sl;
                }
                if (slot < 0) return false;
                g.cc[r][slot] += c;
            }
        }
    }
    const int esz = dtype == TP_F32 ? 4 : 2;
    const int w_bytes = T.wnum * esz, g_bytes = T.dim_out * 4, shn = T.dim_sh;
    const int per_edge = w_bytes + g_bytes + shn * 4 + 8;
    const int target = tu.bwd_stage_bytes ? tu.bwd_stage_bytes : 9000;
    int eps = target / per_edge;
    eps = eps < 1 ? 1 : (eps > 10 ? 10 : eps);  // lanes 0..9 and 10..19 issue the rows
    const int ms = cpt >= 2 ? 2 * TP.R : TP.R;
    g.tab_bytes = round_up(24 * TP.R, 128);
    auto layout = [&](int S, int e) {
        g.S = S;
        g.eps = e;
        g.g_off = e * w_bytes;
        g.sh_off = g.g_off + e * g_bytes;
        g.id_off = g.sh_off + round_up(e * shn * 4, 16);
        g.stage_bytes = round_up(g.id_off + e * 8, 128);
        g.m_off = S * g.stage_bytes;
        g.bar_off = round_up(g.m_off + e * ms * 4, 16);
        g.warp_bytes = round_up(g.bar_off + S * 8, 128);
        return g.tab_bytes + g.warp_bytes <= smem_optin;
    };
    // Two stages: one chunk lands while the warp works on the other. The
    // kernel needs ~255 registers a thread, so at most 8 warps fit an SM, and
    // with two stages all 8 also fit its shared memory at the largest rows;
    // measured on the 128-channel, 13-path graph, 8 warps of 2 stages beat 6 of
    // 3 by 1.3x (the ring is latency-bound at this occupancy, not by copies
    // in flight). A ring that does not fit one warp's share shrinks: fewer
    // edges per chunk, then fewer stages.
    int S = tu.bwd_stages ? tu.bwd_stages : 2;
    while (!layout(S, eps) && (eps > 1 || S > 2)) {
        if (eps > 1) --eps;
        else --S;
    }
    int wpb = tu.bwd_warps ? tu.bwd_warps : kRingMaxWarps;
    while (wpb > 1 && g.tab_bytes + wpb * g.warp_bytes > smem_optin) --wpb;
    bl.smem = g.tab_bytes + wpb * g.warp_bytes;
    if (bl.smem > smem_optin) return false;
    bl.wpb = wpb;
    if (cudaFuncSetAttribute(bl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bl.smem) != cudaSuccess) return false;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bl.occ, bl.fn, 32 * wpb, bl.smem) != cudaSuccess ||
        bl.occ < 1)
        return false;
    return true;
}

struct BwdKey {
    uint64_t uid;
    int dev, dtype;
    uint32_t gen;
    bool operator<(const BwdKey &o) const {
        return std::tie(uid, dev, dtype, gen) < std::tie(o.uid, o.dev, o.dtype, o.gen);
    }
};
std::mutex g_bwd_mu;
std::map<BwdKey, std::unique_ptr<BwdLaunch>> g_bwd_plans;  // nullptr: no ring kernel for this key

const BwdLaunch *cached_bwd_plan(const tp_desc *d, tp_dtype dtype, int dev, int smem_optin, const TuningState &ts) {
    const BwdKey key{d->uid, dev, (int)dtype, ts.gen};
    std::lock_guard<std::mutex> lk(g_bwd_mu);
    auto it = g_bwd_plans.find(key);
    if (it != g_bwd_plans.end()) return it->second.get();
    std::unique_ptr<BwdLaunch> bl(new BwdLaunch());
    if (!bwd_plan(d, dtype, smem_optin, ts.t, *bl)) bl.reset();
    const BwdLaunch *p = bl.get();
    g_bwd_plans[key] = std::move(bl);
    return p;
}

// every resident warp slot, but at least ~4 edges per warp (on a small graph
// more warps keep more chunks in flight at once)
void bwd_geometry(const BwdLaunch &bl, int64_t E, int sms, int &n_warps) {
    long long nw = (long long)sms * bl.occ * bl.wpb;
    const long long by_edges = (E + 3) / 4;
    if (nw > by_edges) nw = by_edges;
    if (nw < 1) nw = 1;
    n_warps = (int)nw;
}

}  // namespace

void bwd_cache_forget(uint64_t uid) {
    std::lock_guard<std::mutex> lk(g_bwd_mu);
    for (auto it = g_bwd_plans.begin(); it != g_bwd_plans.end();)
        it = it->first.uid == uid ? g_bwd_plans.erase(it) : std::next(it);
}

size_t ring_bwd_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin) {
    const TuningState ts = tuning_snapshot();
    if (E >= (int64_t)1 << 31) return 0;
    const BwdLaunch *bl = cached_bwd_plan(d, dtype, dev, smem_optin, ts);
    if (!bl) return 0;
    int nw;
    bwd_geometry(*bl, E, sms, nw);
    return bwd_carry_bytes(nw, d->tab.dim_x);
}

cudaError_t ring_backward(const tp_desc *d, tp_dtype dtype, const float *grad_out, const void *x, const float *sh,
                          const void *w, const int32_t *src, const int32_t *dst, const int32_t *src_perm,
                          const int32_t *src_row_ptr, int32_t N_src, int32_t N_dst, int64_t E, float *dx, float *dw,
                          float *dsh, void *ws, size_t ws_bytes, int dev, int sms, int smem_optin, int *status, cudaStream_t stream) {
    const TuningState ts = tuning_snapshot();
    if (!ws || E >= (int64_t)1 << 31) return cudaErrorNotSupported;
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                         reinterpret_cast<uintptr_t>(grad_out) | reinterpret_cast<uintptr_t>(dx) |
                         reinterpret_cast<uintptr_t>(dw);
    if ((al & 15u) != 0 || (reinterpret_cast<uintptr_t>(sh) & 3u) || (reinterpret_cast<uintptr_t>(dsh) & 3u))
        return cudaErrorNotSupported;
    const BwdLaunch *bl = cached_bwd_plan(d, dtype, dev, smem_optin, ts);
    if (!bl) return cudaErrorNotSupported;
    const Tables &T = d->tab;
    int n_warps;
    bwd_geometry(*bl, E, sms, n_warps);
    while (n_warps > 1 && bwd_carry_bytes(n_warps, T.dim_x) > ws_bytes) n_warps = (n_warps + 1) / 2;
    if (bwd_carry_bytes(n_warps, T.dim_x) > ws_bytes) return cudaErrorNotSupported;
    static_assert(sizeof(RingBwdParams) < 32000, "kernel parameter block too large");
    RingBwdParams prm = bl->geo;
    prm.x = x;
    prm.g = grad_out;
    prm.sh = sh;
    prm.w = w;
    prm.src = src;
    prm.dst = dst;
    prm.perm = src_perm;
    prm.row_ptr = src_row_ptr;
    prm.dx = dx;
    prm.dw = dw;
    prm.dsh = dsh;
    prm.carry = static_cast<float *>(ws);
    const size_t cb = ((size_t)2 * n_warps * T.dim_x * sizeof(float) + 255) / 256 * 256;
    prm.carry_dst = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + cb);
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.n_warps = n_warps;
    prm.n_pieces = n_warps;
    prm.E = E;
    prm.wait_ns = ts.t.wait_limit_ns > 0 ? (uint64_t)ts.t.wait_limit_ns : kWaitNs;
    const int blocks = (n_warps + bl->wpb - 1) / bl->wpb;
    void *args[] = {&prm};
    cudaError_t e = cudaLaunchKernel(bl->fn, dim3(blocks), dim3(32 * bl->wpb), args, (size_t)bl->smem, stream);
    if (e != cudaSuccess) return e;
    const int wpb = 8;
    carry_fixup_kernel<<<(n_warps + wpb - 1) / wpb, 32 * wpb, 0, stream>>>(prm.carry, prm.carry_dst, n_warps, T.dim_x,
                                                                         N_src, dx);
    return cudaGetLastError();
}

}  // namespace tpc
