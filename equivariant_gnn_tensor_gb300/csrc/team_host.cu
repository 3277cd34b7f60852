// Host side of the program-specialised forward: launch geometry, workspace
// for the head/tail partials of destinations cut by stream boundaries, and the
// partial-merging kernel.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "direct_fwd.cuh"
#include "team_fwd.cuh"

namespace tpc {

const void *team_kernel_f32(int shape, int cpt);
const void *team_kernel_bf16(int shape, int cpt);
const void *direct_kernel_f32(int shape, int cpt);
const void *direct_kernel_bf16(int shape, int cpt);

__global__ void carry_fixup_kernel(const float *__restrict__ carry, const int32_t *__restrict__ carry_dst,
                                   int n_streams, int dim_out, float *__restrict__ out) {
    const int c = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (c >= n_streams) return;
    const int d = carry_dst[2 * c + 1];
    if (d < 0) return;
    for (int col = lane * 4; col < dim_out; col += 128) {
        float4 v = *reinterpret_cast<const float4 *>(carry + (int64_t)(2 * c + 1) * dim_out + col);
        for (int c2 = c + 1; c2 < n_streams && carry_dst[2 * c2] == d; ++c2) {
            const float4 u = *reinterpret_cast<const float4 *>(carry + (int64_t)(2 * c2) * dim_out + col);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
        *reinterpret_cast<float4 *>(out + (int64_t)d * dim_out + col) = v;
    }
}

struct TeamLaunch {
    const void *fn = nullptr;
    TeamLayout L{};
    int consumers = 0, cpt = 0, streams = 0, smem = 0;
};

static int env_int(const char *name, int dflt) {
    const char *v = std::getenv(name);
    return v && *v ? std::atoi(v) : dflt;
}

static size_t carry_bytes(int streams, int dim_out) {
    const size_t a = (size_t)2 * streams * dim_out * sizeof(float);
    return (a + 255) / 256 * 256 + (size_t)2 * streams * sizeof(int32_t);
}

// Plan the launch; returns false when the descriptor has no program kernel.
// `sms`/`smem_optin` describe the current device.
static bool team_plan(const tp_desc *d, tp_dtype dtype, int64_t E, int sms, int smem_optin, TeamLaunch &tl) {
    const TeamPlan &TP = d->team;
    if (!TP.valid) return false;
    const int mul = d->tab.mul;
    int cpt = env_int("TPCONV_TEAM_CPT", mul >= 128 ? 1 : 1);
    if (cpt != 1 && cpt != 2) cpt = 1;
    if (mul % (32 * cpt) != 0) cpt = 1;
    if (mul % 32 != 0) return false;
    const int cs = mul / (32 * cpt);
    if (cs < 1 || cs > kTeamMaxConsumers) return false;
    tl.fn = dtype == TP_F32 ? team_kernel_f32(TP.shape, cpt) : team_kernel_bf16(TP.shape, cpt);
    if (!tl.fn) return false;
    const int esz = dtype == TP_F32 ? 4 : 2;
    TeamLayout &L = tl.L;
    L.w_bytes = d->tab.wnum * esz;
    L.f_bytes = d->tab.dim_x * esz;
    L.sh_floats = d->tab.dim_sh;
    const int per_edge = L.w_bytes + L.f_bytes + L.sh_floats * 4;
    int eps = env_int("TPCONV_TEAM_STAGE_BYTES", 6144) / per_edge;
    eps = eps < 1 ? 1 : (eps > 8 ? 8 : eps);
    L.S = env_int("TPCONV_TEAM_STAGES", 3);
    if (L.S < 2 || L.S > kTeamMaxStages) L.S = 4;
    L.eps = eps;
    L.R = TP.R;
    L.nnz = TP.nnz;
    L.w_off = 0;
    L.f_off = eps * L.w_bytes;
    L.sh_off = L.f_off + eps * L.f_bytes;
    L.stage_bytes = round_up(L.sh_off + eps * L.sh_floats * 4, 128);
    L.tab_off = 0;
    L.bar_off = 0;
    L.meta_off = L.bar_off + 3 * L.S * 8;
    L.stage_off = round_up(L.meta_off + L.S * (int)sizeof(ChunkMeta), 128);
    L.m_off = L.stage_off + L.S * L.stage_bytes;
    L.total = round_up(L.m_off + L.S * eps * L.R * 4, 128);
    if (L.total > smem_optin) return false;
    tl.consumers = cs;
    tl.cpt = cpt;
    tl.smem = L.total;
    int occ = 0;
    if (cudaFuncSetAttribute(tl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess) return false;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, tl.fn, 32 * (cs + 1), L.total) != cudaSuccess || occ < 1)
        return false;
    long long streams = (long long)sms * occ;
    const long long by_edges = (E + 31) / 32;
    if (streams > by_edges) streams = by_edges;
    if (streams < 1) streams = 1;
    tl.streams = (int)streams;
    return true;
}

struct DirectLaunch {
    const void *fn = nullptr;
    int cs = 0, cpt = 0, streams = 0, blocks = 0, smem = 0, S = 0, slot_words = 0;
};
constexpr int kDirectWarps = 8;

static bool direct_plan(const tp_desc *d, tp_dtype dtype, int64_t E, int sms, DirectLaunch &dl) {
    const TeamPlan &TP = d->team;
    if (!TP.valid) return false;
    const int mul = d->tab.mul;
    if (mul % 32 != 0) return false;
    // bfloat16 rows are copied in 4-byte pairs: at least two channels per lane
    const int cpt_min = dtype == TP_F32 ? 1 : 2;
    int cpt = env_int("TPCONV_DIRECT_CPT", cpt_min);
    if (cpt != 1 && cpt != 2) cpt = cpt_min;
    if (cpt < cpt_min) cpt = cpt_min;
    if (mul % (32 * cpt) != 0) return false;
    const int cs = mul / (32 * cpt);
    if (cs < 1 || cs > kDirectWarps || kDirectWarps % cs != 0) return false;
    dl.fn = dtype == TP_F32 ? direct_kernel_f32(TP.shape, cpt) : direct_kernel_bf16(TP.shape, cpt);
    if (!dl.fn) return false;
    dl.cs = cs;
    dl.cpt = cpt;
    const ProgShape shp = kProgShapes[TP.shape];
    const int np = make_natural_program(shp.li, shp.lsh, shp.lo).n;
    const int ri = (shp.li + 1) * (shp.li + 1);
    const int wpl = dtype == TP_F32 ? cpt : cpt / 2;
    if (wpl < 1) return false;
    dl.slot_words = (np + ri) * 32 * wpl + 64;
    dl.S = env_int("TPCONV_DIRECT_STAGES", 4);
    if (dl.S < 2 || dl.S > 8) dl.S = 4;
    dl.smem = kDirectWarps * (TP.R + dl.S * dl.slot_words) * (int)sizeof(float);
    if (cudaFuncSetAttribute(dl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dl.smem) != cudaSuccess) return false;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dl.fn, 32 * kDirectWarps, dl.smem) != cudaSuccess || occ < 1)
        return false;
    long long streams = (long long)sms * occ * kDirectWarps / cs;
    const long long by_edges = (E + 31) / 32;
    if (streams > by_edges) streams = by_edges;
    if (streams < 1) streams = 1;
    dl.streams = (int)streams;
    dl.blocks = (int)((streams * cs + kDirectWarps - 1) / kDirectWarps);
    return true;
}

// Kernel choice: rows of 32 channels (one warp per stream, small per-edge
// rows) stream best through the per-warp ring; wider rows through the CTA
// pipeline whose consumers split the channels. TPCONV_FWD_PIPELINED=0/1 forces
// one or the other.
static bool use_direct(const tp_desc *d) {
    const int forced = env_int("TPCONV_FWD_PIPELINED", -1);
    if (forced == 0) return true;
    if (forced == 1) return false;
    return d->tab.mul <= 32;
}

size_t team_workspace_bytes(const tp_desc *d, tp_dtype dtype, int64_t E, int sms, int smem_optin) {
    if (use_direct(d)) {
        DirectLaunch dl;
        if (!direct_plan(d, dtype, E, sms, dl)) return 0;
        return carry_bytes(dl.streams, d->tab.dim_out);
    }
    TeamLaunch tl;
    if (!team_plan(d, dtype, E, sms, smem_optin, tl)) return 0;
    return carry_bytes(tl.streams, d->tab.dim_out);
}

static cudaError_t direct_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                                  const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst,
                                  int64_t E, float *out, void *ws, size_t ws_bytes, int sms, int *status,
                                  cudaStream_t stream) {
    DirectLaunch dl;
    if (!direct_plan(d, dtype, E, sms, dl)) return cudaErrorNotSupported;
    int streams = dl.streams;
    while (streams > 0 && carry_bytes(streams, d->tab.dim_out) > ws_bytes) streams >>= 1;
    if (streams < 1 || !ws) return cudaErrorNotSupported;
    static_assert(sizeof(DirectParams) < 32000, "kernel parameter block too large");
    DirectParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const Tables &T = d->tab;
    prm.mul = T.mul;
    prm.dim_x = T.dim_x;
    prm.dim_sh = T.dim_sh;
    prm.dim_out = T.dim_out;
    prm.wnum = T.wnum;
    prm.cs = dl.cs;
    prm.S = dl.S;
    prm.slot_floats = dl.slot_words;
    for (int l = 0; l < 4; ++l) {
        prm.x_off[l] = T.x_off[l];
        prm.o_off[l] = T.o_off[l];
    }
    std::memcpy(prm.wofs, d->team.wofs, sizeof(prm.wofs));
    std::memcpy(prm.ej, d->team.ej, sizeof(uint32_t) * d->team.R);
    std::memcpy(prm.ec, d->team.ec, sizeof(float) * 2 * d->team.R);
    prm.x = x;
    prm.sh = sh;
    prm.w = w;
    prm.src = src;
    prm.row_ptr = row_ptr;
    prm.out = out;
    prm.carry = static_cast<float *>(ws);
    const size_t cb = ((size_t)2 * streams * T.dim_out * sizeof(float) + 255) / 256 * 256;
    prm.carry_dst = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + cb);
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.n_streams = streams;
    prm.E = E;
    const int blocks = (streams * dl.cs + kDirectWarps - 1) / kDirectWarps;
    void *args[] = {&prm};
    cudaError_t e = cudaLaunchKernel(dl.fn, dim3(blocks), dim3(32 * kDirectWarps), args, (size_t)dl.smem, stream);
    if (e != cudaSuccess) return e;
    const int wpb = 8;
    carry_fixup_kernel<<<(streams + wpb - 1) / wpb, 32 * wpb, 0, stream>>>(prm.carry, prm.carry_dst, streams,
                                                                            T.dim_out, out);
    return cudaGetLastError();
}

// Launches the program kernel (+ partial merge). Returns cudaErrorNotSupported
// when the descriptor has no program kernel or the workspace cannot hold one
// stream's partials (the caller then uses the generic kernel).
cudaError_t team_forward(const tp_desc *d, tp_dtype dtype, const void *x, const float *sh, const void *w,
                         const int32_t *src, const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                         float *out, void *ws, size_t ws_bytes, int sms, int smem_optin, int *status,
                         cudaStream_t stream) {
    if (env_int("TPCONV_DISABLE_TEAM", 0)) return cudaErrorNotSupported;
    if (use_direct(d))
        return direct_forward(d, dtype, x, sh, w, src, row_ptr, N_src, N_dst, E, out, ws, ws_bytes, sms, status,
                              stream);
    TeamLaunch tl;
    if (!team_plan(d, dtype, E, sms, smem_optin, tl)) return cudaErrorNotSupported;
    int streams = tl.streams;
    while (streams > 0 && carry_bytes(streams, d->tab.dim_out) > ws_bytes) streams >>= 1;
    if (streams < 1 || !ws) return cudaErrorNotSupported;
    static_assert(sizeof(TeamParams) < 32000, "kernel parameter block too large");
    TeamParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.L = tl.L;
    const Tables &T = d->tab;
    prm.mul = T.mul;
    prm.dim_x = T.dim_x;
    prm.dim_sh = T.dim_sh;
    prm.dim_out = T.dim_out;
    prm.wnum = T.wnum;
    prm.consumers = tl.consumers;
    prm.copy_mode = env_int("TPCONV_TEAM_COPY", 0);
    for (int l = 0; l < 4; ++l) {
        prm.x_off[l] = T.x_off[l];
        prm.o_off[l] = T.o_off[l];
    }
    std::memcpy(prm.wofs, d->team.wofs, sizeof(prm.wofs));
    std::memcpy(prm.ej, d->team.ej, sizeof(uint32_t) * d->team.R);
    std::memcpy(prm.ec, d->team.ec, sizeof(float) * 2 * d->team.R);
    prm.x = x;
    prm.sh = sh;
    prm.w = w;
    prm.src = src;
    prm.row_ptr = row_ptr;
    prm.out = out;
    prm.carry = static_cast<float *>(ws);
    const size_t cb = ((size_t)2 * streams * T.dim_out * sizeof(float) + 255) / 256 * 256;
    prm.carry_dst = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + cb);
    prm.status = status;
    prm.n_src = N_src;
    prm.n_dst = N_dst;
    prm.n_streams = streams;
    prm.E = E;
    void *args[] = {&prm};
    cudaError_t e = cudaLaunchKernel(tl.fn, dim3(streams), dim3(32 * (tl.consumers + 1)), args, (size_t)tl.smem, stream);
    if (e != cudaSuccess) return e;
    const int wpb = 8;
    carry_fixup_kernel<<<(streams + wpb - 1) / wpb, 32 * wpb, 0, stream>>>(prm.carry, prm.carry_dst, streams,
                                                                            T.dim_out, out);
    return cudaGetLastError();
}

}  // namespace tpc
