// Forward kernel for irreps shapes with a compile-time path program
// (program.h), built for memory-level parallelism: every warp streams its own
// edges S-1 edges ahead of the arithmetic into a warp-private shared-memory
// ring with 4-byte cp.async copies, laid out so that each lane later reads back
// exactly the elements it copied itself (so its own cp.async.wait_group is the
// only synchronisation the ring needs), and many warps per SM keep HBM busy.
// No producer warp, no barriers between warps.
//
// Work split: the destination-sorted edge list is cut into `n_streams` exact,
// contiguous, equal shares. A stream is handled by CS warps that split the
// channels (CPT per lane) and walk the same edges. Per edge a warp
//   1. issues the copies of edge e+S-1 into the ring, waits for edge e's
//      slot and reads its weight-row slice, gathered x-row slice and harmonic;
//   2. builds the edge's matrices M_p[i][k] = sum_j C_p[i,j,k] sh[j] (each lane
//      a few entries, at most two terms each, harmonics broadcast by shuffles)
//      into a per-warp shared buffer;
//   3. runs every path of the program as straight-line FMAs into the
//      destination row held in registers.
// When the destination changes the row is stored, or - for a destination cut
// by a stream boundary - written as a head/tail partial that the merge kernel
// (carry_fixup_kernel) adds in stream order. No atomics: results are bitwise
// reproducible for a given device.
#pragma once
#include "team_fwd.cuh"

namespace tpc {

struct DirectParams {
    int32_t mul, dim_x, dim_sh, dim_out, wnum, cs;
    int32_t S;          // ring slots per warp
    int32_t slot_floats;  // 32-bit words per slot
    int32_t x_off[4], o_off[4];
    int16_t wofs[kProgMaxPaths];
    uint32_t ej[kMaxM];
    float ec[kMaxM][2];
    const void *x;
    const float *sh;
    const void *w;
    const int32_t *src;
    const int32_t *row_ptr;
    float *out;
    float *carry;
    int32_t *carry_dst;
    int *status;
    int32_t n_src, n_dst, n_streams;
    int64_t E;
};

// Contraction of one program path with the weights already in registers.
template <int LI, int LSH, int LO, int T, int CPT>
__device__ __forceinline__ void direct_path(float (&acc)[rows_upto(LO)][CPT], const float (&xr)[rows_upto(LI)][CPT],
                                            const float (&wv)[CPT], const float *Mq) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int LA = P.p[T].la, LC = P.p[T].lc;
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NZ = P.nz[T], MO = P.moff[T];
    constexpr int NZ4 = (NZ + 3) / 4;
    float m[NZ4 * 4];
    const float4 *M4 = reinterpret_cast<const float4 *>(Mq + MO);
#pragma unroll
    for (int q = 0; q < NZ4; ++q) {
        const float4 t = M4[q];
        m[4 * q] = t.x;
        m[4 * q + 1] = t.y;
        m[4 * q + 2] = t.z;
        m[4 * q + 3] = t.w;
    }
    if constexpr (NA <= NC) {
        float wx[NA][CPT];
#pragma unroll
        for (int i = 0; i < NA; ++i)
#pragma unroll
            for (int c = 0; c < CPT; ++c) wx[i][c] = wv[c] * xr[LA * LA + i][c];
        static_for<NZ>([&](auto qc) {
            constexpr int code = P.ik[T][decltype(qc)::value];
            constexpr int i = code >> 3, k = code & 7;
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[LC * LC + k][c] = fmaf(m[decltype(qc)::value], wx[i][c], acc[LC * LC + k][c]);
        });
    } else {
        float tk[NC][CPT];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int c = 0; c < CPT; ++c) tk[k][c] = 0.f;
        static_for<NZ>([&](auto qc) {
            constexpr int code = P.ik[T][decltype(qc)::value];
            constexpr int i = code >> 3, k = code & 7;
#pragma unroll
            for (int c = 0; c < CPT; ++c) tk[k][c] = fmaf(m[decltype(qc)::value], xr[LA * LA + i][c], tk[k][c]);
        });
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[LC * LC + k][c] = fmaf(wv[c], tk[k][c], acc[LC * LC + k][c]);
    }
}

template <int LI, int LSH, int LO, int CPT, typename FT>
__global__ void __launch_bounds__(256) direct_fwd_kernel(const __grid_constant__ DirectParams prm) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int RI = rows_upto(LI), RO = rows_upto(LO);
    constexpr int NP = P.n;
    constexpr int KR = (P.R + 31) / 32;
    extern __shared__ __align__(16) float dsm[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    float *Mq = dsm + wib * P.R;  // this warp's M buffer
    const int gw = blockIdx.x * (blockDim.x >> 5) + wib;
    const int CS = prm.cs;
    const int stream = gw / CS, g = gw - stream * CS;
    const int nS = prm.n_streams;
    if (stream >= nS) return;
    const int mul = prm.mul;
    const int ch0 = (g * 32 + lane) * CPT;
    const int64_t E = prm.E;
    const int N = prm.n_dst;
    const int32_t *rp = prm.row_ptr;
    const int64_t e_lo = (int64_t)stream * E / nS, e_hi = (int64_t)(stream + 1) * E / nS;

    // destination range of this stream (same rule as the pipelined kernel)
    int d_start = warp_first_geq(rp, N, e_lo, lane);
    if (d_start > N) d_start = N;
    if (d_start > 0 && (int64_t)rp[d_start] > e_lo) d_start -= 1;
    int d_end = stream == nS - 1 ? N : warp_first_geq(rp, N, e_hi, lane);
    if (d_end > N) d_end = N;
    if (d_end < d_start) d_end = d_start;
    const int head_dst = (d_start < d_end && (int64_t)rp[d_start] < e_lo) ? d_start : -1;
    int tail_dst = (stream < nS - 1 && d_end > d_start && (int64_t)rp[d_end] > e_hi) ? d_end - 1 : -1;
    if (tail_dst == head_dst) tail_dst = -1;
    if (g == 0 && lane == 0) {
        prm.carry_dst[2 * stream] = head_dst;
        prm.carry_dst[2 * stream + 1] = tail_dst;
    }

    // this lane's M entries and their terms
    uint32_t rj[KR];
    float rc0[KR], rc1[KR];
#pragma unroll
    for (int k = 0; k < KR; ++k) {
        const int r = lane + 32 * k;
        rj[k] = r < P.R ? prm.ej[r] : 0u;
        rc0[k] = r < P.R ? prm.ec[r][0] : 0.f;
        rc1[k] = r < P.R ? prm.ec[r][1] : 0.f;
    }

    // row_ptr window (lane l holds rp[wbase + l]) and src windows
    int wbase = d_start;
    int32_t wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
    auto rp_get = [&](int d) -> int64_t {
        if (d < wbase || d >= wbase + 32) {
            wbase = d;
            wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
        }
        return (int64_t)__shfl_sync(0xffffffffu, wv, d - wbase);
    };
    int64_t sbase = e_lo;
    int sw0 = (sbase + lane < e_hi) ? prm.src[sbase + lane] : 0;
    int sw1 = (sbase + 32 + lane < e_hi) ? prm.src[sbase + 32 + lane] : 0;
    auto src_of = [&](int64_t e) {  // warp-uniform e
        const int off = (int)(e - sbase);
        const int v0 = __shfl_sync(0xffffffffu, sw0, off & 31);
        const int v1 = __shfl_sync(0xffffffffu, sw1, off & 31);
        return off < 32 ? v0 : v1;
    };
    auto src_advance = [&](int64_t e_next) {
        while (e_next >= sbase + 32) {
            sbase += 32;
            sw0 = sw1;
            sw1 = (sbase + 32 + lane < e_hi) ? prm.src[sbase + 32 + lane] : 0;
        }
    };

    const FT *xp = static_cast<const FT *>(prm.x);
    const FT *wp = static_cast<const FT *>(prm.w);
    const int shn = prm.dim_sh;
    float acc[RO][CPT];
#pragma unroll
    for (int r = 0; r < RO; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;

    auto store_row = [&](int d) {
        float *orow;
        if (d == head_dst) orow = prm.carry + (int64_t)(2 * stream) * prm.dim_out;
        else if (d == tail_dst) orow = prm.carry + (int64_t)(2 * stream + 1) * prm.dim_out;
        else orow = prm.out + (int64_t)d * prm.dim_out;
#pragma unroll
        for (int l = 0; l <= LO; ++l) {
            const int off = prm.o_off[l];
            if (off < 0) continue;
#pragma unroll
            for (int k = 0; k < 2 * l + 1; ++k) store_vec<CPT>(orow + off + k * mul + ch0, acc[l * l + k]);
        }
#pragma unroll
        for (int r = 0; r < RO; ++r)
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;
    };

    // Ring slot layout (32-bit words, lane-private columns):
    //   [t*32*WPL + lane*WPL + v]            weight words of path t
    //   [(NP + r)*32*WPL + lane*WPL + v]     x words of row r
    //   [(NP + RI)*32*WPL + lane]            harmonic component `lane`
    //   [(NP + RI)*32*WPL + 32 + lane]       1 if the edge's source index is valid
    // WPL = words per lane per row (CPT floats, or CPT/2 packed bf16 pairs).
    constexpr int WPL = sizeof(FT) == 4 ? CPT : CPT / 2;
    static_assert(WPL >= 1, "bfloat16 rows need at least two channels per lane");
    const int S = prm.S;
    uint32_t *ring = reinterpret_cast<uint32_t *>(dsm + (blockDim.x >> 5) * P.R) + (size_t)wib * S * prm.slot_floats;
    auto issue_edge = [&](int64_t e, int slot) {
        uint32_t *sl = ring + slot * prm.slot_floats;
        const FT *wrow = wp + e * prm.wnum + ch0;
#pragma unroll
        for (int t = 0; t < NP; ++t)
#pragma unroll
            for (int v = 0; v < WPL; ++v) cp_async4(sl + t * 32 * WPL + lane * WPL + v, reinterpret_cast<const uint32_t *>(wrow + prm.wofs[t]) + v);
        const int s = src_of(e);
        const bool okx = s >= 0 && s < prm.n_src;
        sl[(NP + RI) * 32 * WPL + 32 + lane] = okx ? 1u : 0u;
        if (okx) {
            const FT *xrow = xp + (int64_t)s * prm.dim_x + ch0;
#pragma unroll
            for (int l = 0; l <= LI; ++l)
#pragma unroll
                for (int i = 0; i < 2 * l + 1; ++i)
#pragma unroll
                    for (int v = 0; v < WPL; ++v)
                        cp_async4(sl + (NP + l * l + i) * 32 * WPL + lane * WPL + v,
                                  reinterpret_cast<const uint32_t *>(xrow + prm.x_off[l] + i * mul) + v);
        }
        if (lane < shn) cp_async4(sl + (NP + RI) * 32 * WPL + lane, prm.sh + e * shn + lane);
    };
    auto read_vec = [&](const uint32_t *p, float (&v)[CPT]) {
        if constexpr (sizeof(FT) == 4) {
#pragma unroll
            for (int c = 0; c < CPT; ++c) v[c] = __uint_as_float(p[c]);
        } else {
#pragma unroll
            for (int c = 0; c < CPT / 2; ++c) {
                v[2 * c] = bf16lo(p[c]);
                v[2 * c + 1] = bf16hi(p[c]);
            }
        }
    };

    int cur_d = d_start;
    int64_t seg_end = 0;
    auto enter = [&](int d) {
        if (d >= d_end) return;
        int64_t a = rp_get(d), b = rp_get(d + 1);
        if (a < 0 || b < a || b > E) {
            if (lane == 0) set_status(prm.status, TP_DEV_ERR_SEGMENT);
            b = a < 0 ? 0 : (a > E ? E : a);
        }
        seg_end = b < e_hi ? b : e_hi;
    };
    enter(cur_d);
    // prologue: edges e_lo .. e_lo+S-2 in flight (one commit group per slot, empty groups past the end)
    int64_t e_iss = e_lo;
    for (int k = 0; k < S - 1; ++k) {
        if (e_iss < e_hi) {
            src_advance(e_iss);
            issue_edge(e_iss, k);
        }
        ++e_iss;
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    int slot = 0;
    for (int64_t e = e_lo; e < e_hi; ++e) {
        // close destinations that end before edge e (including empty ones)
        while (cur_d < d_end && e >= seg_end) {
            store_row(cur_d);
            ++cur_d;
            enter(cur_d);
        }
        // keep S-1 edges in flight: issue edge e+S-1 into the slot freed last iteration
        {
            const int islot = slot == 0 ? S - 1 : slot - 1;
            if (e_iss < e_hi) {
                src_advance(e_iss);
                issue_edge(e_iss, islot);
            }
            ++e_iss;
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        // wait until at most S-1 groups are pending: edge e's group has landed
        cp_async_wait_pending(S - 1);
        const uint32_t *sl = ring + slot * prm.slot_floats;
        float wc[NP][CPT], xc[RI][CPT];
#pragma unroll
        for (int t = 0; t < NP; ++t) read_vec(sl + t * 32 * WPL + lane * WPL, wc[t]);
#pragma unroll
        for (int r = 0; r < RI; ++r) read_vec(sl + (NP + r) * 32 * WPL + lane * WPL, xc[r]);
        const float shc = lane < shn ? __uint_as_float(sl[(NP + RI) * 32 * WPL + lane]) : 0.f;
        const bool ok = sl[(NP + RI) * 32 * WPL + 32 + lane] != 0u;
        if (!ok && lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
        // M for edge e
#pragma unroll
        for (int k = 0; k < KR; ++k) {
            const float s0 = __shfl_sync(0xffffffffu, shc, rj[k] & 0xffffu);
            const float s1 = __shfl_sync(0xffffffffu, shc, rj[k] >> 16);
            const int r = lane + 32 * k;
            if (r < P.R) Mq[r] = fmaf(rc0[k], s0, rc1[k] * s1);
        }
        __syncwarp();
        if (ok) {
            static_for<NP>([&](auto tc) {
                constexpr int T = decltype(tc)::value;
                direct_path<LI, LSH, LO, T, CPT>(acc, xc, wc[T], Mq);
            });
        }
        __syncwarp();
        slot = slot + 1 == S ? 0 : slot + 1;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // close the rest (last destination, and trailing empty ones on the last stream)
    while (cur_d < d_end) {
        store_row(cur_d);
        ++cur_d;
    }
}

}  // namespace tpc
