// Warp-per-segment convolution kernel: one warp owns whole segments (a
// destination row, or a source row for the input gradient), streams the
// segment's edges through a private multi-stage shared-memory pipeline filled
// by the TMA bulk-copy engine (weight rows, gathered feature rows) and
// cp.async (harmonic rows), and keeps per-segment state in registers. No
// atomics and a fixed summation order: results are bitwise reproducible.
//
// kFwd      segments = destinations; slot t is edge t of the destination-sorted
//           list; gathers x[src[e]]; a chunk's weight rows are contiguous (one
//           bulk copy); accumulates out[d] in registers.
// kBwdX     segments = sources; slot t is edge src_perm[t]; gathers
//           grad_out[dst[e]]; weight rows gathered one bulk copy per edge;
//           accumulates dx[s] in registers.
// kBwdEdge  segments = destinations as in kFwd; keeps grad_out[d] in registers
//           and writes dw[e] and dsh[e] for every edge (per-lane partial sums of
//           the harmonic gradient are reduced across the warp through shared
//           memory).
#pragma once
#include "conv_common.cuh"

namespace tpc {

enum ConvMode { kFwd = 0, kBwdX = 1, kBwdEdge = 2 };

struct SegParams {
    Tables tab;
    WarpLayout lay;
    const void *feat;         // gathered rows (x for kFwd/kBwdEdge, grad_out for kBwdX)
    const float *sh;          // [E][dim_sh]
    const void *w;            // [E][wnum]
    const int32_t *gidx;      // per edge: row of `feat` to gather (src, or dst for kBwdX)
    const int32_t *seg_ptr;   // [n_seg+1]
    const int32_t *slot_edge; // kBwdX: edge of each slot (src_perm); otherwise unused
    const float *g;           // kBwdEdge: grad_out [n_seg][dim_out]
    float *out;               // kFwd: out [n_seg][dim_out]; kBwdX: dx [n_seg][dim_x]
    float *dw;                // kBwdEdge: [E][wnum]
    float *dsh;               // kBwdEdge: [E][dim_sh]
    int *status;
    int32_t n_seg;            // segments
    int32_t n_gather;         // rows of feat
    int64_t n_edges;
    uint64_t wait_ns;         // main-loop pipeline wait limit
};

template <int LI, int LO, int CPT, typename FT, int MODE>
__global__ void __launch_bounds__(256, 1) seg_conv_kernel(const __grid_constant__ SegParams prm) {
    constexpr int RI = rows_upto(LI), RO = rows_upto(LO);
    constexpr int RF = MODE == kBwdX ? RO : RI;  // rows of the gathered feature
    constexpr int RA = MODE == kBwdX ? RI : RO;  // rows of the register row (acc, or grad_out for kBwdEdge)
    constexpr int LF = MODE == kBwdX ? LO : LI;
    constexpr int LA_ = MODE == kBwdX ? LI : LO;
    extern __shared__ __align__(128) unsigned char smem[];
    const Tables &T = prm.tab;
    const WarpLayout &L = prm.lay;
    SmemTables *st = reinterpret_cast<SmemTables *>(smem);
    SmemTrTables *tt = reinterpret_cast<SmemTrTables *>(smem + kTablesBytes);
    for (int q = threadIdx.x; q <= T.R; q += blockDim.x) st->rec_ptr[q] = T.rec_ptr[q];
    for (int q = threadIdx.x; q < T.nnz; q += blockDim.x) {
        st->rec_j[q] = T.rec_j[q];
        st->rec_c[q] = T.rec_c[q];
    }
    if constexpr (MODE == kBwdEdge) {
        for (int q = threadIdx.x; q <= T.dim_sh; q += blockDim.x) tt->tr_ptr[q] = T.tr_ptr[q];
        for (int q = threadIdx.x; q < T.nnz; q += blockDim.x) {
            tt->tr_r[q] = T.tr_r[q];
            tt->tr_c[q] = T.tr_c[q];
        }
    }
    constexpr int kHead = kTablesBytes + (MODE == kBwdEdge ? kTrTablesBytes : 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    unsigned char *wbase = smem + kHead + warp * L.warp_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
    ChunkMeta *meta = reinterpret_cast<ChunkMeta *>(wbase + 8 * L.stages);
    unsigned char *stages = wbase + L.head_bytes;
    float *Ms = reinterpret_cast<float *>(stages + L.stages * L.stage_bytes);
    float *Qs = Ms + L.m_floats;     // kBwdEdge: [R][33] lane partials
    float *Qf = Qs + T.R * 33;       // kBwdEdge: [R] reduced
    if (lane == 0)
        for (int s = 0; s < L.stages; ++s) mbar_init(&bars[s], 33);
    fence_barrier_init();
    __syncthreads();

    const int mul = T.mul;
    const int fdim = MODE == kBwdX ? T.dim_out : T.dim_x;
    const int ch0 = lane * CPT;
    const bool active = ch0 < mul;
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const FT *featp = static_cast<const FT *>(prm.feat);
    const FT *wp = static_cast<const FT *>(prm.w);
    const int W = gridDim.x * nwarps;
    const int64_t E = prm.n_edges;

    // ---- chunk iterator (warp-uniform) ---------------------------------
    int it_seg = blockIdx.x * nwarps + warp;
    int it_e = 0, it_end = 0;
    bool it_first = true;
    int nx_start = 0, nx_end = 0;  // bounds of segment it_seg + W (prefetched)
    auto load_bounds = [&](int s, int &a, int &b) {
        if (s < prm.n_seg) {
            a = prm.seg_ptr[s];
            b = prm.seg_ptr[s + 1];
        } else {
            a = b = 0;
        }
    };
    auto check_bounds = [&](int &a, int &b) {
        if (a < 0 || b < a || (int64_t)b > E) {
            set_status(prm.status, TP_DEV_ERR_SEGMENT);
            a = b = 0;
        }
    };
    load_bounds(it_seg, it_e, it_end);
    check_bounds(it_e, it_end);
    load_bounds(it_seg + W, nx_start, nx_end);

    auto take = [&]() {
        ChunkMeta m;
        if (it_seg >= prm.n_seg) {
            m.seg = -1;
            m.e0 = 0;
            m.n = 0;
            m.bits = 0;
            return m;
        }
        m.seg = it_seg;
        m.e0 = it_e;
        m.n = min(L.eps, it_end - it_e);
        m.bits = kValid | (it_first ? kFirst : 0u);
        it_e += m.n;
        it_first = false;
        if (it_e >= it_end) {
            m.bits |= kLast;
            it_seg += W;
            it_e = nx_start;
            it_end = nx_end;
            check_bounds(it_e, it_end);
            it_first = true;
            load_bounds(it_seg + W, nx_start, nx_end);
        }
        return m;
    };

    // pending chunk and its per-lane indices (loaded one chunk ahead)
    ChunkMeta pend = take();
    int p_edge = 0, p_row = -1;
    auto load_idx = [&](const ChunkMeta &m, int &edge, int &row) {
        edge = -1;
        row = -1;
        if ((m.bits & kValid) && lane < m.n) {
            if constexpr (MODE == kBwdX) edge = prm.slot_edge[m.e0 + lane];
            else edge = m.e0 + lane;
            if (edge >= 0 && edge < E) row = prm.gidx[edge];
            else edge = -1;
        }
    };
    load_idx(pend, p_edge, p_row);

    auto issue = [&](int s) {
        ChunkMeta m = pend;
        int edge = p_edge, row = p_row;
        // advance the iterator and start the next chunk's index loads now
        pend = take();
        load_idx(pend, p_edge, p_row);
        if (!(m.bits & kValid)) {
            if (lane == 0) meta[s] = m;
            return false;
        }
        const bool ok = lane < m.n && edge >= 0 && row >= 0 && row < prm.n_gather;
        const bool bad = lane < m.n && !ok;
        if (__any_sync(0xffffffffu, bad)) set_status(prm.status, TP_DEV_ERR_INDEX);
        const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
        unsigned char *sb = stages + s * L.stage_bytes;
        float *shs = reinterpret_cast<float *>(sb + L.sh_off);
        const int shn = L.sh_floats;
        if constexpr (MODE != kBwdX) {
            const float *shsrc = prm.sh + (int64_t)m.e0 * shn;
            for (int q = lane; q < m.n * shn; q += 32) cp_async4(shs + q, shsrc + q);
        } else {
            for (int q = 0; q < m.n; ++q) {
                const int eq = __shfl_sync(0xffffffffu, edge, q);
                if (eq >= 0)
                    for (int j = lane; j < shn; j += 32) cp_async4(shs + q * shn + j, prm.sh + (int64_t)eq * shn + j);
            }
        }
        cp_async_mbar_arrive_noinc(&bars[s]);
        uint32_t bytes = (uint32_t)__popc(okmask) * (uint32_t)L.f_bytes;
        if constexpr (MODE != kBwdX) bytes += (uint32_t)m.n * (uint32_t)L.w_bytes;
        else bytes += (uint32_t)__popc(okmask) * (uint32_t)L.w_bytes;
        if (lane == 0) {
            ChunkMeta mm = m;
            mm.bits |= okmask << 8;
            meta[s] = mm;
            mbar_arrive_expect_tx(&bars[s], bytes);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if constexpr (MODE != kBwdX) {
            if (lane == 0 && m.n > 0)
                bulk_g2s(sb + L.w_off, wp + (int64_t)m.e0 * T.wnum, (uint32_t)(m.n * L.w_bytes), &bars[s], pol_stream);
        } else {
            if (ok)
                bulk_g2s(sb + L.w_off + lane * L.w_bytes, wp + (int64_t)edge * T.wnum, (uint32_t)L.w_bytes, &bars[s],
                         pol_stream);
        }
        if (ok)
            bulk_g2s(sb + L.f_off + lane * L.f_bytes, featp + (int64_t)row * fdim, (uint32_t)L.f_bytes, &bars[s],
                     pol_keep);
        return true;
    };

    uint32_t phase = 0;     // bit s = parity of the next wait on stage s
    uint32_t inflight = 0;  // bit s = stage s holds an issued chunk
    for (int s = 0; s < L.stages; ++s)
        if (issue(s)) inflight |= 1u << s;

    // per-segment register row: accumulator (kFwd, kBwdX) or grad_out[d] (kBwdEdge)
    float acc[RA][CPT];
#pragma unroll
    for (int r = 0; r < RA; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;

    bool failed = false;
    for (int s = 0;; s = (s + 1 == L.stages) ? 0 : s + 1) {
        if (!((inflight >> s) & 1u)) break;
        const bool ok = mbar_wait(&bars[s], (phase >> s) & 1u, prm.wait_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
        }
        phase ^= 1u << s;
        const ChunkMeta m = meta[s];
        const unsigned char *sb = stages + s * L.stage_bytes;
        const float *shs = reinterpret_cast<const float *>(sb + L.sh_off);
        build_m(st, shs, L.sh_floats, m.n, T.R, Ms, lane);
        __syncwarp();
        if (m.bits & kFirst) {
            if constexpr (MODE == kBwdEdge) {
                const float *grow = prm.g + (int64_t)m.seg * T.dim_out;
#pragma unroll
                for (int l = 0; l <= LO; ++l) {
                    const int off = T.o_off[l];
#pragma unroll
                    for (int k = 0; k < 2 * l + 1; ++k) {
                        if (off >= 0 && active) load_vec<CPT>(grow + off + k * mul + ch0, acc[l * l + k]);
                        else {
#pragma unroll
                            for (int c = 0; c < CPT; ++c) acc[l * l + k][c] = 0.f;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < RA; ++r)
#pragma unroll
                    for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;
            }
        }
        for (int q = 0; q < m.n; ++q) {
            if (!((m.bits >> (8 + q)) & 1u)) {
                if constexpr (MODE == kBwdEdge) {  // a skipped edge still gets zero gradient rows
                    const int64_t e = m.e0 + q;
                    for (int t = lane; t < T.wnum; t += 32) prm.dw[e * T.wnum + t] = 0.f;
                    for (int j = lane; j < T.dim_sh; j += 32) prm.dsh[e * T.dim_sh + j] = 0.f;
                }
                continue;
            }
            const FT *fs = reinterpret_cast<const FT *>(sb + L.f_off + q * L.f_bytes);
            const FT *ws = reinterpret_cast<const FT *>(sb + L.w_off + q * L.w_bytes);
            const float *Mq = Ms + q * T.R;
            float fr[RF][CPT];
#pragma unroll
            for (int l = 0; l <= LF; ++l) {
                const int off = MODE == kBwdX ? T.o_off[l] : T.x_off[l];
#pragma unroll
                for (int i = 0; i < 2 * l + 1; ++i) {
                    if (off >= 0 && active) {
                        load_vec<CPT>(fs + off + i * mul + ch0, fr[l * l + i]);
                    } else {
#pragma unroll
                        for (int c = 0; c < CPT; ++c) fr[l * l + i][c] = 0.f;
                    }
                }
            }
            const int64_t e = m.e0 + q;  // kBwdEdge: edge id (contiguous)
            for (int p = 0; p < T.n_paths; ++p) {
                float wv[CPT];
                if (active) load_vec<CPT>(ws + p * mul + ch0, wv);
                else {
#pragma unroll
                    for (int c = 0; c < CPT; ++c) wv[c] = 0.f;
                }
                const float *Mp = Mq + T.m_off[p];
                const int key = T.la[p] * 4 + T.lc[p];
                float dwv[CPT];
#define TPC_CASE(A, C)                                                                          \
    case (A)*4 + (C):                                                                           \
        if constexpr ((A) <= LI && (C) <= LO) {                                                 \
            if constexpr (MODE == kFwd) path_fwd<A, C, RI, RO, CPT>(acc, fr, wv, Mp);              \
            else if constexpr (MODE == kBwdX) path_bwd_x<A, C, RI, RO, CPT>(acc, fr, wv, Mp);      \
            else path_bwd_edge<A, C, RI, RO, CPT>(fr, acc, wv, Mp, dwv, Qs + T.m_off[p] * 33 + lane); \
        }                                                                                       \
        break;
                switch (key) {
                    TPC_CASE(0, 0) TPC_CASE(0, 1) TPC_CASE(0, 2) TPC_CASE(0, 3)
                    TPC_CASE(1, 0) TPC_CASE(1, 1) TPC_CASE(1, 2) TPC_CASE(1, 3)
                    TPC_CASE(2, 0) TPC_CASE(2, 1) TPC_CASE(2, 2) TPC_CASE(2, 3)
                    TPC_CASE(3, 0) TPC_CASE(3, 1) TPC_CASE(3, 2) TPC_CASE(3, 3)
                    default: break;
                }
#undef TPC_CASE
                if constexpr (MODE == kBwdEdge) {
                    if (active) store_vec<CPT>(prm.dw + e * T.wnum + p * mul + ch0, dwv);
                }
            }
            if constexpr (MODE == kBwdEdge) {
                // reduce the lane partials of Q, then dsh[j] = sum_r G[r][j] Q[r]
                __syncwarp();
                for (int r = lane; r < T.R; r += 32) {
                    const float *row = Qs + r * 33;
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int l2 = 0; l2 < 32; l2 += 2) {
                        s0 += row[l2];
                        s1 += row[l2 + 1];
                    }
                    Qf[r] = s0 + s1;
                }
                __syncwarp();
                for (int j = lane; j < T.dim_sh; j += 32) {
                    float sacc = 0.f;
                    const int t1 = tt->tr_ptr[j + 1];
                    for (int t = tt->tr_ptr[j]; t < t1; ++t) sacc = fmaf(tt->tr_c[t], Qf[tt->tr_r[t]], sacc);
                    prm.dsh[e * T.dim_sh + j] = sacc;
                }
                __syncwarp();
            }
        }
        if constexpr (MODE != kBwdEdge) {
            if ((m.bits & kLast) && active) {
                const int odim = MODE == kFwd ? T.dim_out : T.dim_x;
                float *orow = prm.out + (int64_t)m.seg * odim;
#pragma unroll
                for (int l = 0; l <= LA_; ++l) {
                    const int off = MODE == kFwd ? T.o_off[l] : T.x_off[l];
                    if (off < 0) continue;
#pragma unroll
                    for (int k = 0; k < 2 * l + 1; ++k) store_vec<CPT>(orow + off + k * mul + ch0, acc[l * l + k]);
                }
            }
        }
        __syncwarp();
        if (issue(s)) inflight |= 1u << s;
        else inflight &= ~(1u << s);
    }
    if (failed) {
        set_status(prm.status, TP_DEV_ERR_TIMEOUT);
        // let copies still in flight land (full time limit) before the block's
        // shared memory is released
        for (int s = 0; s < L.stages; ++s)
            if ((inflight >> s) & 1u) (void)mbar_wait(&bars[s], (phase >> s) & 1u, kWaitNs);
    }
}

}  // namespace tpc
