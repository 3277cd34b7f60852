// Backward kernel for irreps shapes with a compile-time path program
// (program.h), one pass by source: for the upstream gradient g = dL/d out of
// the forward out[d] = sum_{e: dst e = d} sum_p w_p[e] (M_p[e]^T x[src e])
// (channelwise, M_p[e][i][k] = sum_j C_p[i,j,k] sh[e][j]) it computes
//   dx[s]       = sum_{e: src e = s} sum_p w_p[e] (.) (M_p[e] g[dst e])
//   dw_p[e][u]  = sum_{i,k} M_p[e][i][k] x[s][i][u] g[dst e][k][u]
//   dsh[e][j]   = sum_p sum_{i,k} C_p[i,j,k] sum_u w_p[e][u] x[s][i][u] g[dst e][k][u]
// Every edge's weight row is read once and its weight-gradient row written
// once; x[s] is a register row for the whole segment of s, and the gathered
// rows g[dst e] stay in L2.
//
// Work split as in the forward ring kernel: the source-sorted slot list
// (slot t holds edge src_perm[t]) is cut into equal contiguous pieces, piece p
// belongs to warp p % n_warps, and a source cut by a piece boundary is written
// as a head/tail partial row that carry_fixup_kernel adds in piece order.
//
// Per warp, a private S-stage shared-memory ring:
//   issue:   chunks of up to `eps` slots; per edge one bulk (TMA) copy of the
//            weight row (lane q) and one of the gradient row g[dst e]
//            (lane 10 + q), and the harmonic row by cp.async; the slots' edge
//            ids are loaded two chunks ahead and their destinations and
//            sources one chunk ahead, so no copy waits on a dependent index
//            load. An edge whose source is not the segment's (a source CSR
//            that does not match src) or whose destination is out of range is
//            flagged and gets zero dw and dsh rows and no dx term.
//   consume: M of the chunk's edges from the harmonic rows (lane-parallel over
//            entries), then per edge every path as straight-line code:
//              s_i  = sum_k M[i][k] g_k                (lane channels)
//              dw   = sum_i x_i (.) s_i                -> stored
//              dx_i += w (.) s_i                        (registers)
//              h_ik = sum over the lane's channels of w x_i g_k, added with the
//                     entry's Clebsch-Gordan coefficient to the lane's partial
//                     harmonic gradient of each component j that feeds it
//            and after the last path a transposed butterfly over the warp
//            reduces the partial harmonic gradients, one component per lane
//            pair, stored as dsh[e].
// No atomics: results are bitwise reproducible for a given launch geometry.
#pragma once
#include "ring_fwd.cuh"

namespace tpc {

struct RingBwdParams {
    int32_t S, eps;                               // stages per warp, slots per chunk (<= 10)
    int32_t stage_bytes, g_off, sh_off, id_off;   // stage: weight rows at 0, gradient rows, harmonic rows,
                                                  // {edge id, its source} pairs
    int32_t m_off, bar_off, warp_bytes;           // warp region: stages, M, barriers
    int32_t tab_bytes;                            // block-shared: M recipe int4[R], then coefficients float2[R]
    uint32_t ej[kMaxM];                           // M entry r = ec[r][0] * sh[ej & 0xffff] + ec[r][1] * sh[ej >> 16]
    float ec[kMaxM][2];
    float cc[kMaxM][2];                           // coefficient of component m_entry_j(.., slot) in M entry r
    const void *x;
    const float *g;
    const float *sh;
    const void *w;
    const int32_t *src;
    const int32_t *dst;
    const int32_t *perm;     // slot -> edge (src_perm)
    const int32_t *row_ptr;  // source CSR over slots (src_row_ptr)
    float *dx, *dw, *dsh;
    float *carry;            // [2*n_pieces][dim_x]
    int32_t *carry_dst;      // [2*n_pieces]
    int *status;
    int32_t n_src, n_dst, n_warps, n_pieces;
    int64_t E;
    uint64_t wait_ns;
};

// Sum of the lane values of a packed pair (or a single float).
__device__ __forceinline__ float lane_sum(float v) { return v; }
__device__ __forceinline__ float lane_sum(f32x2 v) { return lo_f(v) + hi_f(v); }

// Is entry q of path T the first that reaches input row i of its path?
template <int LI, int LSH, int LO>
constexpr bool first_of_i(int T, int q) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    for (int q2 = 0; q2 < q; ++q2)
        if ((P.ik[T][q2] >> 3) == (P.ik[T][q] >> 3)) return false;
    return true;
}
// Smallest input row of path T that some entry reaches.
template <int LI, int LSH, int LO>
constexpr int min_i(int T) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    int m = 99;
    for (int q = 0; q < P.nz[T]; ++q) m = (P.ik[T][q] >> 3) < m ? (P.ik[T][q] >> 3) : m;
    return m;
}

// Harmonic component (index in the harmonic row) `slot` of entry q of path T, or -1.
template <int LI, int LSH, int LO, int T>
constexpr int bwd_j(int q, int slot) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    const int j = m_entry_j(P.p[T].la, P.p[T].lb, P.p[T].lc, P.ik[T][q] >> 3, P.ik[T][q] & 7, slot);
    return j < 0 ? -1 : P.p[T].lb * P.p[T].lb + j;
}

// One program path of one edge. xr: x[s] (lane channels); wl, gl: this lane's
// channels of the edge's staged weight and gradient rows; Mq: the edge's M
// (entries duplicated into pairs for channel pairs); cct: per-entry
// coefficients of the components feeding it; dacc: the lane's partial
// harmonic gradient; dwl: this lane's channels of the edge's dw row.
template <int LI, int LSH, int LO, int T, int CPT, bool PK, typename FT, int SHP>
__device__ __forceinline__ void bwd_path(typename LaneVec<CPT, PK>::V (&acc)[rows_upto(LI)][LaneVec<CPT, PK>::NV],
                                         const typename LaneVec<CPT, PK>::V (&xr)[rows_upto(LI)][LaneVec<CPT, PK>::NV],
                                         const FT *wl, const float *gl, const float *Mq, const float2 *cct,
                                         float (&dacc)[SHP], float *dwl) {
    using LV = LaneVec<CPT, PK>;
    using V = typename LV::V;
    constexpr int NV = LV::NV;
    constexpr int MUL = 32 * CPT;
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int LA = P.p[T].la, LC = P.p[T].lc;
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NZ = P.nz[T], MO = P.moff[T];
    V wv[NV];
    load_lane<CPT, PK>(wl + T * MUL, wv);
    V gk[NC][NV];
    static_for<NC>([&](auto kc) {
        constexpr int k = decltype(kc)::value;
        if constexpr (has_k<LI, LSH, LO>(T, k)) load_lane<CPT, PK>(gl + (LC * LC + k) * MUL, gk[k]);
    });
    // s_i = sum_k M[i][k] g_k
    V s[NA][NV];
    static_for<NZ>([&](auto qc) {
        constexpr int q = decltype(qc)::value;
        constexpr int i = P.ik[T][q] >> 3, k = P.ik[T][q] & 7;
        constexpr bool first = first_of_i<LI, LSH, LO>(T, q);
        V m;
        if constexpr (LV::kPair) m = *reinterpret_cast<const f32x2 *>(Mq + 2 * (MO + q));
        else m = Mq[MO + q];
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            if constexpr (first) s[i][c] = vmul(m, gk[k][c]);
            else vfma(s[i][c], m, gk[k][c]);
        }
    });
    // harmonic gradient partials: h_ik = sum_lane (w x_i) g_k
    V wx[NA][NV];
    static_for<NA>([&](auto ic) {
        constexpr int i = decltype(ic)::value;
        if constexpr (has_i<LI, LSH, LO>(T, i)) {
#pragma unroll
            for (int c = 0; c < NV; ++c) wx[i][c] = vmul(wv[c], xr[LA * LA + i][c]);
        }
    });
    static_for<NZ>([&](auto qc) {
        constexpr int q = decltype(qc)::value;
        constexpr int i = P.ik[T][q] >> 3, k = P.ik[T][q] & 7;
        constexpr int J0 = bwd_j<LI, LSH, LO, T>(q, 0), J1 = bwd_j<LI, LSH, LO, T>(q, 1);
        static_assert(J0 >= 0 && J0 < SHP && J1 < SHP, "pattern entry without a harmonic component");
        V p = vmul(wx[i][0], gk[k][0]);
#pragma unroll
        for (int c = 1; c < NV; ++c) vfma(p, wx[i][c], gk[k][c]);
        const float h = lane_sum(p);
        const float2 cq = cct[MO + q];
        dacc[J0] = fmaf(cq.x, h, dacc[J0]);
        if constexpr (J1 >= 0) dacc[J1] = fmaf(cq.y, h, dacc[J1]);
    });
    // dw = sum_i x_i (.) s_i; dx_i += w (.) s_i
    static_assert(NZ > 0, "a program path has at least one entry");
    V dwv[NV];
    static_for<NA>([&](auto ic) {
        constexpr int i = decltype(ic)::value;
        if constexpr (has_i<LI, LSH, LO>(T, i)) {
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                if constexpr (i == min_i<LI, LSH, LO>(T)) dwv[c] = vmul(xr[LA * LA + i][c], s[i][c]);
                else vfma(dwv[c], xr[LA * LA + i][c], s[i][c]);
                vfma(acc[LA * LA + i][c], wv[c], s[i][c]);
            }
        }
    });
    store_lane<CPT, PK>(dwl + T * MUL, dwv);
}

// SHP partial sums per lane -> their sums over the warp; afterwards lane l
// holds the total of component l >> (5 - log2 SHP) in v[0].
template <int SHP>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[SHP], int lane) {
    int width = SHP, off = 16;
#pragma unroll
    for (; width > 1; width >>= 1, off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int t = 0; t < SHP / 2; ++t) {
            if (t < width / 2) {
                const float send = up ? v[t] : v[t + width / 2];
                const float keep = up ? v[t + width / 2] : v[t];
                v[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}

template <int LI, int LSH, int LO, int CPT, bool PK, typename FT>
__global__ void __launch_bounds__(32 * kRingMaxWarps, 1) ring_bwd_kernel(const __grid_constant__ RingBwdParams prm) {
    using LV = LaneVec<CPT, PK>;
    using V = typename LV::V;
    constexpr int NV = LV::NV;
    static_assert(!LV::kEdgePair, "the backward packs channel pairs only");
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int RI = rows_upto(LI), RO = rows_upto(LO), SHN = rows_upto(LSH);
    constexpr int KR = (P.R + 31) / 32;
    constexpr int MUL = 32 * CPT;
    constexpr int DX = RI * MUL, DOUT = RO * MUL;
    constexpr int WNUM = P.n * MUL;
    constexpr int WB = WNUM * (int)sizeof(FT), GB = DOUT * 4;
    constexpr int MS = LV::kPair ? 2 * P.R : P.R;
    constexpr int SHP = SHN <= 4 ? 4 : (SHN <= 8 ? 8 : 16);
    constexpr int SHL = SHP == 4 ? 2 : (SHP == 8 ? 3 : 4);
    static_assert(WB % 16 == 0 && GB % 16 == 0, "bulk copies move 16-byte multiples");
    extern __shared__ __align__(128) unsigned char smem[];
    int4 *tab = reinterpret_cast<int4 *>(smem);
    float2 *cct = reinterpret_cast<float2 *>(smem + 16 * P.R);
    for (int r = threadIdx.x; r < P.R; r += blockDim.x) {
        tab[r] = make_int4((int)(prm.ej[r] & 0xffffu) * 4, (int)(prm.ej[r] >> 16) * 4, __float_as_int(prm.ec[r][0]),
                           __float_as_int(prm.ec[r][1]));
        cct[r] = make_float2(prm.cc[r][0], prm.cc[r][1]);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int gw = blockIdx.x * (blockDim.x >> 5) + wib;
    if (gw >= prm.n_warps) return;
    const int S = prm.S, eps = prm.eps;
    unsigned char *base = smem + prm.tab_bytes + (size_t)wib * prm.warp_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + prm.bar_off);
    float *Mw = reinterpret_cast<float *>(base + prm.m_off);
    // 32 cp.async arrivals (harmonic rows) + the expect-tx arrival per phase
    if (lane == 0)
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 33);
    fence_barrier_init();
    __syncwarp();

    const int nP = prm.n_pieces, nW = prm.n_warps, N = prm.n_src;
    const int E = (int)prm.E;  // the host launches this kernel only for E < 2^31
    const int32_t *rp = prm.row_ptr;
    const int32_t *permp = prm.perm;
    const int32_t *dstp = prm.dst;
    const int32_t *srcp = prm.src;
    const FT *xp = static_cast<const FT *>(prm.x);
    const unsigned char *wb = static_cast<const unsigned char *>(prm.w);
    const float *gp = prm.g;
    const int ch0 = lane * CPT;
    auto piece_lo = [&](int p) -> int { return (int)((int64_t)p * E / nP); };

    // ---- issue side --------------------------------------------------------------
    struct Cur {
        int p, e, hi, n;
    };
    auto settle = [&](Cur &c) {
        while (c.p < nP && c.e >= c.hi) {
            c.p += nW;
            if (c.p < nP) {
                c.e = piece_lo(c.p);
                c.hi = piece_lo(c.p + 1);
            }
        }
        c.n = c.p < nP ? min(eps, c.hi - c.e) : 0;
    };
    auto advance = [](Cur c) {
        c.e += c.n;
        return c;
    };
    // edge id of slot c.e + lane (-1 when absent or out of range)
    auto load_edge = [&](const Cur &c) -> int {
        if (lane >= c.n) return -1;
        const int e = permp[c.e + lane];
        return (uint32_t)e < (uint32_t)E ? e : -2;  // -2: flagged when the chunk is issued
    };
    auto load_dst = [&](int e) -> int { return e >= 0 ? dstp[e] : -1; };
    auto load_src = [&](int e) -> int { return e >= 0 ? srcp[e] : -1; };
    Cur ic{gw, gw < nP ? piece_lo(gw) : 0, gw < nP ? piece_lo(gw + 1) : 0, 0};
    settle(ic);
    Cur lc = advance(ic);
    settle(lc);
    Cur mc = advance(lc);
    settle(mc);
    int eA = load_edge(ic), eB = load_edge(lc), eC = load_edge(mc);
    int dA = load_dst(eA), dB = load_dst(eB);
    int sA = load_src(eA), sB = load_src(eB);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int n_issued = 0, s_iss = 0;
    auto issue_next = [&]() {
        const int n = ic.n;
        if (n == 0) return;
        const int s = s_iss;
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        unsigned char *sb = base + s * prm.stage_bytes;
        const bool ev = lane < n && eA >= 0;
        const bool dv = ev && (uint32_t)dA < (uint32_t)prm.n_dst;
        const uint32_t evm = __ballot_sync(0xffffffffu, ev), dvm = __ballot_sync(0xffffffffu, dv);
        if (__any_sync(0xffffffffu, (lane < n && !ev) || (ev && !dv)) && lane == 0)
            set_status(prm.status, TP_DEV_ERR_INDEX);
        if (lane < n) reinterpret_cast<int2 *>(sb + prm.id_off)[lane] = make_int2(ev ? eA : -1, sA);
        // an edge whose destination is out of range gets a zero gradient row:
        // its weight and harmonic gradients come out zero, its dx term too
        if (evm != dvm)
            for (int q = 0; q < n; ++q)
                if (((evm & ~dvm) >> q) & 1u)
                    for (int o = lane * 16; o < GB; o += 512)
                        *reinterpret_cast<uint4 *>(sb + prm.g_off + q * GB + o) = make_uint4(0, 0, 0, 0);
        // harmonic rows by cp.async, 4 bytes at a time (a warp-uniform loop:
        // every lane takes part in each shuffle)
        float *shs = reinterpret_cast<float *>(sb + prm.sh_off);
        for (int t0 = 0; t0 < n * SHN; t0 += 32) {
            const int t = t0 + lane;
            const int q = t < n * SHN ? t / SHN : 0, j = t - q * SHN;
            const int eq = __shfl_sync(0xffffffffu, eA, q);
            if (t < n * SHN && (uint32_t)eq < (uint32_t)E) cp_async4(shs + t, prm.sh + (int64_t)eq * SHN + j);
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(evm) * WB + (uint32_t)__popc(dvm) * GB);
        cp_async_mbar_arrive_noinc(&full[s]);
        __syncwarp();
        // lane q < 10: weight row of edge q; lane 10 + q: gradient row of edge q
        const int q = lane < 10 ? lane : lane - 10;
        const int eq = __shfl_sync(0xffffffffu, eA, q & 31);
        const int dq = __shfl_sync(0xffffffffu, dA, q & 31);
        if (lane < 10 && q < n && ((evm >> q) & 1u))
            bulk_g2s(sb + q * WB, wb + (int64_t)eq * WB, (uint32_t)WB, &full[s], pol_stream);
        else if (lane >= 10 && lane < 20 && q < n && ((dvm >> q) & 1u))
            bulk_g2s(sb + prm.g_off + q * GB, gp + (int64_t)dq * DOUT, (uint32_t)GB, &full[s], pol_keep);
        if (lane == 0 && mc.e + 16 * eps < E) asm volatile("prefetch.global.L2 [%0];" ::"l"(permp + mc.e + 16 * eps));
        ++n_issued;
        ic = lc;
        eA = eB;
        dA = dB;
        sA = sB;
        lc = mc;
        eB = eC;
        dB = load_dst(eB);
        sB = load_src(eB);
        mc = advance(mc);
        settle(mc);
        eC = load_edge(mc);
    };
    for (int k = 0; k < S; ++k) issue_next();

    // ---- source ranges of this warp's pieces (as the forward's destination ranges) ----
    const int np_w = gw < nP ? (nP - 1 - gw) / nW + 1 : 0;
    int fb = 0;
    if (np_w == 1) {
        const int f0 = warp_first_geq(rp, N, piece_lo(gw), lane);
        const int f1 = warp_first_geq(rp, N, piece_lo(gw + 1), lane);
        fb = lane == 0 ? f0 : f1;
    } else if (lane < 2 * np_w) {
        fb = lane_first_geq(rp, N, piece_lo(gw + (lane >> 1) * nW + (lane & 1)));
    }
    const int rb = lane < 2 * np_w ? rp[min(fb, N)] : 0;
    auto piece_dstart = [&](int j) {
        const int e_lo = piece_lo(gw + j * nW);
        int d = min(__shfl_sync(0xffffffffu, fb, 2 * j), N);
        const bool earlier = d > 0 && __shfl_sync(0xffffffffu, rb, 2 * j) > e_lo;
        return earlier ? -(d - 1) - 1 : d;
    };

    // ---- consume side -----------------------------------------------------------------
    V acc[RI][NV], xr[RI][NV];
#pragma unroll
    for (int r = 0; r < RI; ++r)
#pragma unroll
        for (int c = 0; c < NV; ++c) acc[r][c] = V(0);
    int n_done = 0, s_done = 0;
    uint32_t ph_done = 0;
    bool failed = false;
    for (int j = 0; j < np_w && !failed; ++j) {
        const int p = gw + j * nW;
        const int e_lo = piece_lo(p), e_hi = piece_lo(p + 1);
        const int ds = piece_dstart(j);
        const int d_start = ds < 0 ? -ds - 1 : ds;
        int d_end = __shfl_sync(0xffffffffu, fb, 2 * j + 1);
        const int rp_end = __shfl_sync(0xffffffffu, rb, 2 * j + 1);
        if (p == nP - 1 || d_end > N) d_end = N;
        if (d_end < d_start) d_end = d_start;
        const int head_dst = (ds < 0 && d_start < d_end) ? d_start : -1;
        int tail_dst = (p < nP - 1 && d_end > d_start && rp_end > e_hi) ? d_end - 1 : -1;
        if (tail_dst == head_dst) tail_dst = -1;
        if (lane == 0) {
            prm.carry_dst[2 * p] = head_dst;
            prm.carry_dst[2 * p + 1] = tail_dst;
        }
        int wbase = d_start;
        int32_t wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
        auto rp_get = [&](int d) -> int {
            if (d < wbase || d >= wbase + 32) {
                wbase = d;
                wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
            }
            return __shfl_sync(0xffffffffu, wv, d - wbase);
        };
        int cur_d = d_start;
        int seg_end = 0;
        auto enter = [&](int d) {
            if (d >= d_end) return;
            const int a = rp_get(d);
            int b = rp_get(d + 1);
            if (a < 0 || b < a || b > E) {
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_SEGMENT);
                b = a < 0 ? 0 : (a > E ? E : a);
            }
            seg_end = b < e_hi ? b : e_hi;
            if (b > a) {  // the source's own row, for every edge of its segment
                const FT *xs = xp + (int64_t)d * DX + ch0;
#pragma unroll
                for (int r = 0; r < RI; ++r) load_lane<CPT, PK>(xs + r * MUL, xr[r]);
            }
        };
        auto store_row = [&](int d) {
            float *orow;
            if (d == head_dst) orow = prm.carry + (int64_t)(2 * p) * DX;
            else if (d == tail_dst) orow = prm.carry + (int64_t)(2 * p + 1) * DX;
            else orow = prm.dx + (int64_t)d * DX;
            orow += ch0;
#pragma unroll
            for (int r = 0; r < RI; ++r) store_lane<CPT, PK>(orow + r * MUL, acc[r]);
#pragma unroll
            for (int r = 0; r < RI; ++r)
#pragma unroll
                for (int c = 0; c < NV; ++c) acc[r][c] = V(0);
        };
        enter(cur_d);
        int e = e_lo;
        while (e < e_hi) {
            const int s = s_done;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph_done, prm.wait_ns))) {
                if (lane == 0) {
                    set_status(prm.status, TP_DEV_ERR_TIMEOUT);
                    for (int j2 = j; j2 < np_w; ++j2) {
                        prm.carry_dst[2 * (gw + j2 * nW)] = -1;
                        prm.carry_dst[2 * (gw + j2 * nW) + 1] = -1;
                    }
                }
                failed = true;
                break;
            }
            const int n = min(eps, e_hi - e);
            const unsigned char *sb = base + s * prm.stage_bytes;
            const int2 *ids = reinterpret_cast<const int2 *>(sb + prm.id_off);
            // M of the chunk's edges (lane-parallel over entries)
            {
                const unsigned char *shq = sb + prm.sh_off;
                int4 t[KR];
#pragma unroll
                for (int k = 0; k < KR; ++k) t[k] = (lane + 32 * k < P.R) ? tab[lane + 32 * k] : make_int4(0, 0, 0, 0);
                float *mo = Mw + (LV::kPair ? 2 * lane : lane);
                for (int q = 0; q < n; ++q) {
#pragma unroll
                    for (int k = 0; k < KR; ++k) {
                        if (lane + 32 * k < P.R) {
                            const float v = fmaf(__int_as_float(t[k].z), *reinterpret_cast<const float *>(shq + t[k].x),
                                                 __int_as_float(t[k].w) * *reinterpret_cast<const float *>(shq + t[k].y));
                            if constexpr (LV::kPair) *reinterpret_cast<float2 *>(mo + 64 * k) = make_float2(v, v);
                            else mo[32 * k] = v;
                        }
                    }
                    shq += SHN * 4;
                    mo += MS;
                }
            }
            __syncwarp();
            for (int q = 0; q < n; ++q, ++e) {
                while (e >= seg_end && cur_d < d_end) {
                    store_row(cur_d);
                    ++cur_d;
                    enter(cur_d);
                }
                const int2 idq = ids[q];
                const int eid = idq.x;
                if (eid < 0) continue;  // slot without a valid edge (flagged at issue)
                if (idq.y != cur_d) {   // the edge's source is not this segment's
                    if (lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
                    for (int t = lane; t < WNUM; t += 32) prm.dw[(int64_t)eid * WNUM + t] = 0.f;
                    if (lane < SHN) prm.dsh[(int64_t)eid * SHN + lane] = 0.f;
                    continue;
                }
                const FT *wl = reinterpret_cast<const FT *>(sb + q * WB) + ch0;
                const float *gl = reinterpret_cast<const float *>(sb + prm.g_off + q * GB) + ch0;
                const float *Mq = Mw + q * MS;
                float *dwl = prm.dw + (int64_t)eid * WNUM + ch0;
                float dacc[SHP];
#pragma unroll
                for (int jj = 0; jj < SHP; ++jj) dacc[jj] = 0.f;
                static_for<P.n>([&](auto tc) {
                    bwd_path<LI, LSH, LO, decltype(tc)::value, CPT, PK, FT, SHP>(acc, xr, wl, gl, Mq, cct, dacc, dwl);
                });
                const float v = warp_transpose_sum<SHP>(dacc, lane);
                const int comp = lane >> (5 - SHL);
                if ((lane & ((1 << (5 - SHL)) - 1)) == 0 && comp < SHN) prm.dsh[(int64_t)eid * SHN + comp] = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            issue_next();
            ++n_done;
            if (++s_done == S) {
                s_done = 0;
                ph_done ^= 1u;
            }
        }
        if (failed) break;
        while (cur_d < d_end) {
            store_row(cur_d);
            ++cur_d;
            enter(cur_d);
        }
    }
    if (failed) {
        for (int k = n_done; k < n_issued; ++k) {
            (void)mbar_wait(&full[s_done], ph_done, kWaitNs);
            if (++s_done == S) {
                s_done = 0;
                ph_done ^= 1u;
            }
        }
    }
}

}  // namespace tpc
