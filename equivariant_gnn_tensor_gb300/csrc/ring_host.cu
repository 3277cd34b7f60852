// Host side of the program-specialised forward: launch geometry of the warp
// ring kernel, the workspace for head/tail partial rows of destinations cut by
// piece boundaries, and the partial-merging kernel.
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>

#include "ring_fwd.cuh"
#include "tuning.h"

namespace tpc {

const void *ring_kernel_f32(int shape, int cpt, int pk);
const void *ring_kernel_bf16(int shape, int cpt, int pk);
const void *ring_kernel_vec_f32(int shape, int cpt, int pk);
const void *ring_kernel_vec_bf16(int shape, int cpt, int pk);
const void *ring_kernel_mlp_f32(int shape, int cpt, int pk);

__global__ void carry_fixup_kernel(const float *__restrict__ carry, const int32_t *__restrict__ carry_dst,
                                   int n_pieces, int dim_out, int n_dst, float *__restrict__ out) {
    const int c = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (c >= n_pieces) return;
    const int d = carry_dst[2 * c + 1];
    if (d < 0 || d >= n_dst) return;
    for (int col = lane * 4; col < dim_out; col += 128) {
        float4 v = *reinterpret_cast<const float4 *>(carry + (int64_t)(2 * c + 1) * dim_out + col);
        for (int c2 = c + 1; c2 < n_pieces && carry_dst[2 * c2] == d; ++c2) {
            const float4 u = *reinterpret_cast<const float4 *>(carry + (int64_t)(2 * c2) * dim_out + col);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
        *reinterpret_cast<float4 *>(out + (int64_t)d * dim_out + col) = v;
    }
}

// head and tail partial rows of every piece, then their destination ids
static size_t carry_bytes(int pieces, int dim_out) {
    const size_t a = (size_t)2 * pieces * dim_out * sizeof(float);
    return (a + 255) / 256 * 256 + (size_t)2 * pieces * sizeof(int32_t);
}

// The part of a ring launch that does not depend on the edge count: kernel,
// shared-memory layout, M recipe, warps per block and blocks per SM.
struct RingKernel {
    const void *fn = nullptr;
    RingParams geo{};  // layout fields and M recipe only
    int wpb = 0, smem = 0, occ = 0;
};
struct RingLaunch {
    const void *fn = nullptr;
    const void *fn_vec = nullptr;  // the same kernel taking edge vectors
    RingParams geo{};  // layout fields and M recipe only
    int wpb = 0, smem = 0, occ = 0, rounds = 1;
    // the kernel computing the weight rows by the radial network (float32
    // only; fn null when there is none): the layout above, or with edge pairs
    // its own (no weight rows in the ring, the second layer in shared memory)
    RingKernel mlp;
};

// One warp covers all channels, CPT = mul/32 in {1,2,4} channels per lane,
// for descriptors in the natural layout the kernel is compiled for.
static bool ring_plan(const tp_desc *d, tp_dtype dtype, int smem_optin, const tp_tuning &tu, RingLaunch &rl) {
    const ProgramPlan &TP = d->prog;
    if (!TP.valid) return false;
    const Tables &T = d->tab;
    const int mul = T.mul;
    if (mul % 32 != 0) return false;
    const int cpt = mul / 32;
    if (cpt != 1 && cpt != 2 && cpt != 4) return false;
    // packed FMAs: channel pairs for two channels per lane, edge pairs for one
    // (the two smaller programs; the larger ones run out of registers); four
    // channels per lane keep plain FMAs (shorter dependent latency)
    const int pk = tu.ring_pack ? (tu.ring_pack == 1) : (cpt == 4 ? 0 : (cpt == 2 || TP.shape <= 1));
    // natural layout: block l at l*l*mul, paths in program order
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
    rl.fn = dtype == TP_F32 ? ring_kernel_f32(TP.shape, cpt, pk) : ring_kernel_bf16(TP.shape, cpt, pk);
    rl.fn_vec = dtype == TP_F32 ? ring_kernel_vec_f32(TP.shape, cpt, pk) : ring_kernel_vec_bf16(TP.shape, cpt, pk);
    const void *fn_mlp = dtype == TP_F32 ? ring_kernel_mlp_f32(TP.shape, cpt, pk) : nullptr;
    if (!rl.fn || !rl.fn_vec) return false;
    const int esz = dtype == TP_F32 ? 4 : 2;
    RingParams &g = rl.geo;
    std::memset(&g, 0, sizeof(g));
    const int w_bytes = T.wnum * esz, f_bytes = T.dim_x * esz;
    const int shn = T.dim_sh;
    const int per_edge = w_bytes + f_bytes + shn * 4;
    // about 4.5 KB per chunk and two stages per warp: one chunk lands while the
    // warp works on the other, and enough warps fit on an SM to keep HBM busy
    const int target = tu.ring_stage_bytes ? tu.ring_stage_bytes : 4500;
    int eps = (target + per_edge - 1) / per_edge;
    eps = eps < 1 ? 1 : (eps > 30 ? 30 : eps);  // lanes 2..31 issue the gathered rows
    g.S = tu.ring_stages ? tu.ring_stages : 2;
    g.eps = eps;
    g.f_off = eps * w_bytes;
    g.sh_off = g.f_off + eps * f_bytes;
    g.stage_bytes = round_up(g.sh_off + eps * shn * 4 + 32, 128);  // +32: 16-byte aligned harmonic span
    g.m_off = g.S * g.stage_bytes;
    g.y_off = round_up(g.m_off + eps * TP.R * (pk ? 8 : 4), 16);
    g.h_off = round_up(g.y_off + eps * shn * 4, 16);
    g.bar_off = round_up(g.h_off + eps * kMlpHidden * 4, 16);
    g.warp_bytes = round_up(g.bar_off + g.S * 8, 128);
    g.tab_bytes = round_up(16 * TP.R, 128);
    std::memcpy(g.ej, TP.ej, sizeof(uint32_t) * TP.R);
    std::memcpy(g.ec, TP.ec, sizeof(float) * 2 * TP.R);
    int wpb = tu.ring_warps ? tu.ring_warps : 8;
    while (wpb > 1 && g.tab_bytes + wpb * g.warp_bytes > smem_optin) --wpb;
    rl.smem = g.tab_bytes + wpb * g.warp_bytes;
    if (rl.smem > smem_optin) return false;
    rl.wpb = wpb;
    if (cudaFuncSetAttribute(rl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, rl.smem) != cudaSuccess ||
        cudaFuncSetAttribute(rl.fn_vec, cudaFuncAttributeMaxDynamicSharedMemorySize, rl.smem) != cudaSuccess)
        return false;
    // both variants launch with the geometry of the smaller occupancy
    int occ_v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&rl.occ, rl.fn, 32 * wpb, rl.smem) != cudaSuccess || rl.occ < 1 ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_v, rl.fn_vec, 32 * wpb, rl.smem) != cudaSuccess || occ_v < 1)
        return false;
    if (occ_v < rl.occ) rl.occ = occ_v;
    // a radial-network kernel with a layout of its own: the ring carries the
    // source rows and edge vectors only; eps from the stage target (or the
    // given default), at most eps_max
    auto own_layout = [&](int eps_def, int eps_max, int s_def, int m_bytes_per_edge, int h_fixed, int h_per_edge,
                          int blk_extra) {
        RingKernel &m = rl.mlp;
        RingParams &h = m.geo;
        h = g;
        const int per_edge_m = f_bytes + 12;
        int em = tu.ring_stage_bytes ? (tu.ring_stage_bytes + per_edge_m - 1) / per_edge_m : eps_def;
        em = em < 1 ? 1 : (em > eps_max ? eps_max : em);
        h.S = tu.ring_stages ? tu.ring_stages : s_def;
        h.eps = em;
        h.f_off = 0;
        h.sh_off = em * f_bytes;
        h.stage_bytes = round_up(h.sh_off + em * 12 + 32, 128);
        h.m_off = h.S * h.stage_bytes;
        h.y_off = round_up(h.m_off + em * m_bytes_per_edge, 16);
        h.h_off = round_up(h.y_off + em * shn * 4, 16);
        h.bar_off = round_up(h.h_off + h_fixed + em * h_per_edge, 16);
        h.warp_bytes = round_up(h.bar_off + h.S * 8, 128);
        h.w2s_off = round_up(16 * TP.R, 128);
        h.tab_bytes = h.w2s_off + blk_extra;
        int wm = tu.ring_warps ? tu.ring_warps : 8;
        while (wm > 1 && h.tab_bytes + wm * h.warp_bytes > smem_optin) --wm;
        m.wpb = wm;
        m.smem = h.tab_bytes + wm * h.warp_bytes;
        if (m.smem <= smem_optin &&
            cudaFuncSetAttribute(fn_mlp, cudaFuncAttributeMaxDynamicSharedMemorySize, m.smem) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&m.occ, fn_mlp, 32 * wm, m.smem) == cudaSuccess &&
            m.occ >= 1)
            m.fn = fn_mlp;
    };
    if (fn_mlp && cpt == 1 && pk && prog.n <= kMlpMaxPaths) {
        // edge pairs: chunks of up to kMlpChunk edges (the weights of one chunk
        // are formed at once), a third stage against the longer time per
        // chunk, the second layer's copy block-shared; h then the edge lengths
        own_layout(kMlpChunk, kMlpChunk, 3, TP.R * 8, kMlpChunk * (kMlpHidden + 1) * 4, 0, kMlpW2sBytes);
    } else if (fn_mlp && !(cpt == 1 && pk)) {
        // plain lanes or channel pairs: each path's weights formed right before the path; about
        // 13 KB chunks (3 edges for mul 128, 7 warps per block fit: measured
        // 591 us against 610 / 663 / 683 us for 1 / 2 / 4 edges and 635 us for
        // a third stage); h per edge
        const int eps_def = (13000 + f_bytes + 12 - 1) / (f_bytes + 12);
        // M per edge: R floats, or R pairs with channel pairs (entries duplicated)
        own_layout(eps_def < 1 ? 1 : eps_def, 30, 2, TP.R * (pk ? 8 : 4), 0, kMlpHidden * 4, 0);
    } else if (fn_mlp) {
        // otherwise the layout of the other two, at the smallest occupancy of the three
        int occ_m = 0;
        if (cudaFuncSetAttribute(fn_mlp, cudaFuncAttributeMaxDynamicSharedMemorySize, rl.smem) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_m, fn_mlp, 32 * wpb, rl.smem) == cudaSuccess &&
            occ_m >= 1) {
            if (occ_m < rl.occ) rl.occ = occ_m;
            rl.mlp.fn = fn_mlp;
            rl.mlp.geo = g;
            rl.mlp.wpb = rl.wpb;
            rl.mlp.smem = rl.smem;
            rl.mlp.occ = rl.occ;
        }
    }
    rl.rounds = tu.ring_rounds ? tu.ring_rounds : 1;
    return true;
}

// Plans are cached per (descriptor, device, dtype, tuning generation), so a
// forward call makes no CUDA attribute or occupancy query after the first.
namespace {
struct PlanKey {
    uint64_t uid;
    int dev, dtype;
    uint32_t gen;
    bool operator<(const PlanKey &o) const {
        return std::tie(uid, dev, dtype, gen) < std::tie(o.uid, o.dev, o.dtype, o.gen);
    }
};
std::mutex g_plan_mu;
std::map<PlanKey, std::unique_ptr<RingLaunch>> g_plans;  // nullptr: no ring kernel for this key
}  // namespace

void mma_cache_forget(uint64_t uid);
void bwd_cache_forget(uint64_t uid);

void launch_cache_forget(uint64_t uid) {
    mma_cache_forget(uid);
    bwd_cache_forget(uid);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (auto it = g_plans.begin(); it != g_plans.end();) it = it->first.uid == uid ? g_plans.erase(it) : std::next(it);
}

static const RingLaunch *cached_plan(const tp_desc *d, tp_dtype dtype, int dev, int smem_optin, const TuningState &ts) {
    const PlanKey key{d->uid, dev, (int)dtype, ts.gen};
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) return it->second.get();
    std::unique_ptr<RingLaunch> rl(new RingLaunch());
    if (!ring_plan(d, dtype, smem_optin, ts.t, *rl)) rl.reset();
    const RingLaunch *p = rl.get();
    g_plans[key] = std::move(rl);
    return p;
}

// Warps and pieces for E edges: every resident warp slot, but at least ~8
// edges (one or two chunks) per warp. A warp walks its chunks one ring stage
// after another, so on a small graph spreading the edges over more warps keeps
// every chunk in flight at once instead of paying one copy latency per chunk.
static void ring_geometry(int occ, int wpb, int rounds, int64_t E, int sms, int &n_warps, int &n_pieces) {
    long long nw = (long long)sms * occ * wpb;
    const long long by_edges = (E + 7) / 8;
    if (nw > by_edges) nw = by_edges;
    if (nw < 1) nw = 1;
    n_warps = (int)nw;
    n_pieces = n_warps * rounds;
}

// Workspace the split forward needs (0: this descriptor has no program kernel
// or the input does not qualify).
size_t split_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int dev, int sms, int smem_optin) {
    const TuningState ts = tuning_snapshot();
    if (ts.t.disable_split || E >= (int64_t)1 << 31) return 0;
    const RingLaunch *rl = cached_plan(d, dtype, dev, smem_optin, ts);
    if (!rl) return 0;
    int nw, np, nwm = 0, npm = 0;
    ring_geometry(rl->occ, rl->wpb, rl->rounds, E, sms, nw, np);
    if (rl->mlp.fn) ring_geometry(rl->mlp.occ, rl->mlp.wpb, rl->rounds, E, sms, nwm, npm);
    return carry_bytes(np > npm ? np : npm, d->tab.dim_out);
}

// Launches the ring kernel (+ partial merge). Returns cudaErrorNotSupported
// when the descriptor or the pointers do not qualify, or the workspace cannot
// hold the partials (the caller then uses the generic kernel).
// vec_mode 0: `sh` holds harmonic rows [E][dim_sh]; 1 / 2: edge vectors [E][3]
// whose harmonics the kernel evaluates (1: of the unit vector, 2: raw). With
// `mlp` the weight rows come from the radial network of the edge length (w unused).
cudaError_t split_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, int vec_mode,
                          const tp_radial_mlp *mlp, const void *w, const int32_t *src, const int32_t *row_ptr,
                          int32_t N_src, int32_t N_dst, int64_t E, float *out, void *ws, size_t ws_bytes, int dev,
                          int sms, int smem_optin, int *status, cudaStream_t stream) {
    const TuningState ts = tuning_snapshot();
    if (ts.t.disable_split || !ws || E >= (int64_t)1 << 31) return cudaErrorNotSupported;  // 32-bit edge indices inside
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                         reinterpret_cast<uintptr_t>(sh);
    if ((al & 15u) != 0) return cudaErrorNotSupported;
    const RingLaunch *rl = cached_plan(d, dtype, dev, smem_optin, ts);
    if (!rl) return cudaErrorNotSupported;
    if (mlp && (!rl->mlp.fn || vec_mode == 0)) return cudaErrorNotSupported;
    const Tables &T = d->tab;
    const void *fn = mlp ? rl->mlp.fn : (vec_mode ? rl->fn_vec : rl->fn);
    const int occ = mlp ? rl->mlp.occ : rl->occ, wpb_k = mlp ? rl->mlp.wpb : rl->wpb;
    const int smem_k = mlp ? rl->mlp.smem : rl->smem;
    int n_warps, n_pieces;
    ring_geometry(occ, wpb_k, rl->rounds, E, sms, n_warps, n_pieces);
    // a smaller caller workspace: fewer warps
    while (n_warps > 1 && carry_bytes(n_warps * rl->rounds, T.dim_out) > ws_bytes) n_warps = (n_warps + 1) / 2;
    n_pieces = n_warps * rl->rounds;
    if (carry_bytes(n_pieces, T.dim_out) > ws_bytes) return cudaErrorNotSupported;
    static_assert(sizeof(RingParams) < 32000, "kernel parameter block too large");
    RingParams prm = mlp ? rl->mlp.geo : rl->geo;
    prm.x = x;
    prm.sh = sh;
    prm.vec_mode = vec_mode;
    if (mlp) {
        prm.mlp_w1 = mlp->w1;
        prm.mlp_b1 = mlp->b1;
        prm.mlp_w2 = mlp->w2;
        prm.mlp_b2 = mlp->b2;
    }
    prm.w = w;
    prm.src = src;
    prm.row_ptr = row_ptr;
    prm.out = out;
    prm.carry = static_cast<float *>(ws);
    const size_t cb = ((size_t)2 * n_pieces * T.dim_out * sizeof(float) + 255) / 256 * 256;
    prm.carry_dst = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + cb);
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.n_warps = n_warps;
    prm.n_pieces = n_pieces;
    prm.E = E;
    prm.wait_ns = ts.t.wait_limit_ns > 0 ? (uint64_t)ts.t.wait_limit_ns : kWaitNs;
    const int blocks = (n_warps + wpb_k - 1) / wpb_k;
    void *args[] = {&prm};
    cudaError_t e = cudaLaunchKernel(fn, dim3(blocks), dim3(32 * wpb_k), args, (size_t)smem_k, stream);
    if (e != cudaSuccess) return e;
    const int wpb = 8;
    carry_fixup_kernel<<<(n_pieces + wpb - 1) / wpb, 32 * wpb, 0, stream>>>(prm.carry, prm.carry_dst, n_pieces,
                                                                            T.dim_out, N_dst, out);
    return cudaGetLastError();
}

}  // namespace tpc
