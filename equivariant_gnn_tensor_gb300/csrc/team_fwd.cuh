// Forward kernel for irreps shapes that have a compile-time path program
// (program.h): one CTA = one producer warp + CS consumer warps sharing an
// S-stage shared-memory pipeline over an exact, contiguous share of the
// destination-sorted edge list.
//
// Producer warp: finds its destination range by a 32-way search of row_ptr,
//   walks it in chunks of up to `eps` edges (never crossing a destination),
//   issues TMA bulk copies of the chunk's weight rows (one copy) and gathered
//   x rows (one per edge) plus cp.async copies of the harmonic rows, and once a
//   chunk has landed builds its per-edge matrices M (program layout) and marks
//   the stage ready.
// Consumer warps: split the channels (CPT per lane), run every path of the
//   program as straight-line code per edge with the destination row in
//   registers, and store it when the destination ends. A destination cut by a
//   stream boundary is stored as a head/tail partial; a second small kernel
//   adds the partials of each cut destination in stream order. No atomics:
//   results are bitwise reproducible for a given grid.
#pragma once
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "conv_common.cuh"
#include "program.h"

namespace tpc {

constexpr int kTeamMaxStages = 8;
constexpr int kTeamMaxConsumers = 4;
constexpr uint32_t kHead = 8u, kTail = 16u;  // ChunkMeta bits: store to a carry slot

struct TeamLayout {
    int S, eps;
    int w_bytes, f_bytes, sh_floats;
    int stage_bytes, w_off, f_off, sh_off;
    int R, nnz;
    int tab_off, bar_off, meta_off, stage_off, m_off, total;
};

struct TeamParams {
    TeamLayout L;
    int32_t mul, dim_x, dim_sh, dim_out, wnum, consumers;
    int32_t copy_mode;  // 0: TMA bulk copies, 1: 16-byte cp.async from all producer lanes
    int32_t x_off[4], o_off[4];
    int16_t wofs[kProgMaxPaths];
    uint32_t ej[kMaxM];     // M entry r = c0 * sh[ej & 0xffff] + c1 * sh[ej >> 16]
    float ec[kMaxM][2];
    const void *x;
    const float *sh;
    const void *w;
    const int32_t *src;
    const int32_t *row_ptr;
    float *out;
    float *carry;        // [2*n_streams][dim_out]
    int32_t *carry_dst;  // [2*n_streams]
    int *status;
    int32_t n_src, n_dst, n_streams;
    int64_t E;
};

template <int N, class F, int... I>
__device__ __forceinline__ void static_for_impl(F &&f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, class F>
__device__ __forceinline__ void static_for(F &&f) {
    static_for_impl<N>(f, std::make_integer_sequence<int, N>{});
}

// Smallest d in [0, N] with rp[d] >= target (N+1 if none); 32-way search by a
// whole warp. rp must be non-decreasing for a meaningful answer; every access
// stays inside rp[0..N] regardless.
__device__ __forceinline__ int warp_first_geq(const int32_t *rp, int N, int64_t target, int lane) {
    int lo = 0, hi = N + 1;  // answer in [lo, hi]; position hi is known true (or N+1)
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int q = lo + lane * step;
        const bool pr = q >= hi || q > N || (int64_t)rp[q] >= target;
        const uint32_t m = __ballot_sync(0xffffffffu, pr);
        if (m == 0) {
            lo = lo + 31 * step + 1;
        } else {
            const int k = __ffs(m) - 1;
            const int nhi = lo + k * step;
            lo = k == 0 ? lo : lo + (k - 1) * step + 1;
            hi = nhi;
        }
    }
    const int q = lo + lane;
    const bool pr = q >= hi || q > N || (int64_t)rp[q] >= target;
    const uint32_t m = __ballot_sync(0xffffffffu, pr);
    return m ? lo + __ffs(m) - 1 : hi;
}

template <int LI, int LSH, int LO, int T, int CPT, typename FT>
__device__ __forceinline__ void team_path(float (&acc)[rows_upto(LO)][CPT], const float (&xr)[rows_upto(LI)][CPT],
                                          const FT *wrow, const float *Mq, int ch0, int wofs) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int LA = P.p[T].la, LC = P.p[T].lc;
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NZ = P.nz[T], MO = P.moff[T];
    constexpr int NZ4 = (NZ + 3) / 4;
    float wv[CPT];
    load_vec<CPT>(wrow + wofs + ch0, wv);
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
__global__ void __launch_bounds__(32 * (kTeamMaxConsumers + 1)) team_fwd_kernel(const __grid_constant__ TeamParams prm) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int RI = rows_upto(LI), RO = rows_upto(LO);
    extern __shared__ __align__(128) unsigned char smem[];
    const TeamLayout &L = prm.L;
    const int S = L.S;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *ready = full + S;
    uint64_t *empty = ready + S;
    ChunkMeta *meta = reinterpret_cast<ChunkMeta *>(smem + L.meta_off);
    unsigned char *stages = smem + L.stage_off;
    float *Mst = reinterpret_cast<float *>(smem + L.m_off);
    const int CS = prm.consumers;
    if (threadIdx.x == 0)
        for (int s = 0; s < S; ++s) {
            // one arrival per warp: per-thread arrivals on one barrier word serialise
            mbar_init(&full[s], 1);
            mbar_init(&ready[s], 1);
            mbar_init(&empty[s], CS);
        }
    fence_barrier_init();
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t E = prm.E;
    const int nC = prm.n_streams;
    const int cta = blockIdx.x;
    const int mul = prm.mul;

    if (warp == 0) {
        // =========================== producer ===========================
        const int32_t *rp = prm.row_ptr;
        const int N = prm.n_dst;
        const int64_t e_lo = (int64_t)cta * E / nC, e_hi = (int64_t)(cta + 1) * E / nC;
        int d_start = warp_first_geq(rp, N, e_lo, lane);
        if (d_start > N) d_start = N;
        if (d_start > 0 && (int64_t)rp[d_start] > e_lo) d_start -= 1;
        int d_end = cta == nC - 1 ? N : warp_first_geq(rp, N, e_hi, lane);
        if (d_end > N) d_end = N;
        if (d_end < d_start) d_end = d_start;
        int head_dst = (d_start < d_end && (int64_t)rp[d_start] < e_lo) ? d_start : -1;
        int tail_dst = (cta < nC - 1 && d_end > d_start && (int64_t)rp[d_end] > e_hi) ? d_end - 1 : -1;
        if (tail_dst == head_dst) tail_dst = -1;
        if (lane == 0) {
            prm.carry_dst[2 * cta] = head_dst;
            prm.carry_dst[2 * cta + 1] = tail_dst;
        }
        // row_ptr window: lane l holds rp[wbase + l]
        int wbase = d_start;
        int32_t wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
        auto rp_get = [&](int d) -> int64_t {
            if (d < wbase || d >= wbase + 32) {
                wbase = d;
                wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
            }
            return (int64_t)__shfl_sync(0xffffffffu, wv, d - wbase);
        };
        int cur_d = d_start;
        int64_t cur_e = 0, seg_hi = 0;
        bool first = true;
        auto enter = [&](int d) {
            if (d >= d_end) return;
            int64_t a = rp_get(d);
            int64_t b = rp_get(d + 1);
            if (a < 0 || b < a || b > E) {
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_SEGMENT);
                a = b = (a < 0 || a > E) ? 0 : a;
            }
            cur_e = a > e_lo ? a : e_lo;
            seg_hi = b < e_hi ? b : e_hi;
            if (seg_hi < cur_e) seg_hi = cur_e;
            first = true;
        };
        enter(cur_d);
        auto next_chunk = [&]() {
            ChunkMeta m;
            if (cur_d >= d_end) {
                m.seg = -1; m.e0 = 0; m.n = 0; m.bits = 0;
                return m;
            }
            m.seg = cur_d;
            m.e0 = (int32_t)cur_e;
            m.n = (int32_t)min((int64_t)L.eps, seg_hi - cur_e);
            m.bits = kValid | (first ? kFirst : 0u);
            cur_e += m.n;
            first = false;
            if (cur_e >= seg_hi) {
                m.bits |= kLast;
                if (cur_d == head_dst) m.bits |= kHead;
                else if (cur_d == tail_dst) m.bits |= kTail;
                ++cur_d;
                enter(cur_d);
            }
            return m;
        };
        const uint64_t pol_stream = policy_evict_first();
        const uint64_t pol_keep = policy_evict_last();
        // this lane's M entries r = lane + 32k and their (at most two) terms
        constexpr int KR = (P.R + 31) / 32;
        uint32_t rj[KR];
        float rc0[KR], rc1[KR];
#pragma unroll
        for (int k = 0; k < KR; ++k) {
            const int r = lane + 32 * k;
            rj[k] = r < P.R ? prm.ej[r] : 0u;
            rc0[k] = r < P.R ? prm.ec[r][0] : 0.f;
            rc1[k] = r < P.R ? prm.ec[r][1] : 0.f;
        }
        const FT *xp = static_cast<const FT *>(prm.x);
        const FT *wp = static_cast<const FT *>(prm.w);
        // src indices stream in order e_lo, e_lo+1, ...: two 32-edge windows,
        // the second loaded 32 edges before it is needed
        int64_t sbase = e_lo;
        int sw0 = (sbase + lane < e_hi) ? prm.src[sbase + lane] : -1;
        int sw1 = (sbase + 32 + lane < e_hi) ? prm.src[sbase + 32 + lane] : -1;
        auto src_of = [&](int64_t e) {
            const int off = (int)(e - sbase);
            const int v0 = __shfl_sync(0xffffffffu, sw0, off & 31);
            const int v1 = __shfl_sync(0xffffffffu, sw1, off & 31);
            return off < 32 ? v0 : v1;
        };
        auto src_advance = [&](int64_t e_next) {
            while (e_next >= sbase + 32) {
                sbase += 32;
                sw0 = sw1;
                sw1 = (sbase + 32 + lane < e_hi) ? prm.src[sbase + 32 + lane] : -1;
            }
        };
        ChunkMeta pend = next_chunk();
        bool term_issued = false;
        int n_issued = 0;
        auto issue = [&](int s) {
            ++n_issued;
            const ChunkMeta m = pend;
            int srow = -1;
            if (!(m.bits & kValid)) {
                term_issued = true;
            } else {
                srow = src_of((int64_t)m.e0 + lane);
                if (lane >= m.n) srow = -1;
                src_advance((int64_t)m.e0 + m.n);
                pend = next_chunk();
            }
            const bool ok = (m.bits & kValid) && lane < m.n && srow >= 0 && srow < prm.n_src;
            const bool bad = (m.bits & kValid) && lane < m.n && !ok;
            if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
            const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
            unsigned char *sb = stages + s * L.stage_bytes;
            float *shs = reinterpret_cast<float *>(sb + L.sh_off);
            const int shn = L.sh_floats;
            // harmonic rows [e0, e0+n): one bulk copy of the 16-byte aligned span
            // around them; a tail that would run past the array end is copied with
            // plain loads instead. shs[sh_lead + q*shn + j] is component j of edge e0+q.
            const int64_t b0 = (int64_t)m.e0 * shn * 4, b1 = ((int64_t)m.e0 + m.n) * shn * 4;
            const int64_t sh_bytes = E * shn * 4;
            const int64_t a0 = b0 & ~(int64_t)15;
            int64_t a1 = (b1 + 15) & ~(int64_t)15;
            if (a1 > sh_bytes) a1 = sh_bytes & ~(int64_t)15;
            if (a1 < a0) a1 = a0;
            const uint32_t sh_tma = m.n > 0 ? (uint32_t)(a1 - a0) : 0u;
            if (m.n > 0 && a1 < b1) {
                const float *srcf = prm.sh + a1 / 4;
                float *dstf = shs + (a1 - a0) / 4;
                for (int q = lane; q < (int)((b1 - a1) / 4); q += 32) dstf[q] = srcf[q];
            }
            if (prm.copy_mode == 1) {
                // every lane moves 16-byte pieces of the weight rows and of each gathered x row;
                // the range checks only guard against a broken launch (they never fire on valid input)
                const unsigned char *wsrc = reinterpret_cast<const unsigned char *>(wp + (int64_t)m.e0 * prm.wnum);
                const int wb = m.n * L.w_bytes;
                const bool w_in = m.e0 >= 0 && (int64_t)m.e0 + m.n <= E && wb <= L.f_off &&
                                  ((reinterpret_cast<uintptr_t>(wsrc) & 15u) == 0);
                if (w_in)
                    for (int o = lane * 16; o < wb; o += 512) cp_async16(sb + L.w_off + o, wsrc + o);
                else if (lane == 0 && m.n > 0) set_status(prm.status, TP_DEV_ERR_INTERNAL);
                for (int q = 0; q < m.n; ++q) {
                    const int r = __shfl_sync(0xffffffffu, srow, q);
                    if (!((okmask >> q) & 1u)) continue;
                    const unsigned char *xsrc = reinterpret_cast<const unsigned char *>(xp + (int64_t)r * prm.dim_x);
                    if ((reinterpret_cast<uintptr_t>(xsrc) & 15u) != 0 || q >= L.eps) {
                        if (lane == 0) set_status(prm.status, TP_DEV_ERR_INTERNAL);
                        continue;
                    }
                    for (int o = lane * 16; o < L.f_bytes; o += 512)
                        cp_async16(sb + L.f_off + q * L.f_bytes + o, xsrc + o);
                }
            }
            if (prm.copy_mode == 1) cp_async_mbar_arrive_noinc(&full[s]);
            const uint32_t bytes = sh_tma + (prm.copy_mode == 1 ? 0u :
                (uint32_t)__popc(okmask) * (uint32_t)L.f_bytes + (uint32_t)m.n * (uint32_t)L.w_bytes);
            __syncwarp();
            if (lane == 0) {
                ChunkMeta mm = m;
                mm.bits |= okmask << 8;
                mm.seg_lead = (int32_t)((b0 - a0) / 4);
                meta[s] = mm;
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            __syncwarp();
            if (lane == 0 && sh_tma > 0)
                bulk_g2s(shs, reinterpret_cast<const unsigned char *>(prm.sh) + a0, sh_tma, &full[s], pol_stream);
            if (prm.copy_mode == 0) {
                if (lane == 0 && m.n > 0)
                    bulk_g2s(sb + L.w_off, wp + (int64_t)m.e0 * prm.wnum, (uint32_t)(m.n * L.w_bytes), &full[s],
                             pol_stream);
                if (ok)
                    bulk_g2s(sb + L.f_off + lane * L.f_bytes, xp + (int64_t)srow * prm.dim_x, (uint32_t)L.f_bytes,
                             &full[s], pol_keep);
            }
        };
        // Event loop: build M for the oldest landed chunk and refill the stage of
        // the oldest consumed chunk, whichever is possible, so data arrival and
        // stage release never wait on each other.
        for (int s = 0; s < S && !term_issued; ++s) issue(s);
        int n_built = 0;
        bool failed = false;
        uint32_t idle = 0;
        for (;;) {
            bool did = false;
            if (n_built < n_issued) {
                const int s = n_built % S;
                if (__all_sync(0xffffffffu, mbar_test_wait(&full[s], (n_built / S) & 1))) {
                    const ChunkMeta m = meta[s];
                    if (m.bits & kValid) {
                        const float *shs = reinterpret_cast<const float *>(stages + s * L.stage_bytes + L.sh_off) +
                                           m.seg_lead;
                        float *Mq = Mst + s * L.eps * P.R;
                        for (int q = 0; q < m.n; ++q) {
                            const float *shq = shs + q * L.sh_floats;
#pragma unroll
                            for (int k = 0; k < KR; ++k) {
                                const int r = lane + 32 * k;
                                if (r < P.R)
                                    Mq[q * P.R + r] = fmaf(rc0[k], shq[rj[k] & 0xffffu], rc1[k] * shq[rj[k] >> 16]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ready[s]);
                    ++n_built;
                    if (!(m.bits & kValid)) break;  // terminator handed to the consumers
                    did = true;
                }
            }
            if (!term_issued) {
                const int j = n_issued - S;  // chunk that last used the stage to refill
                if (j < n_built && __all_sync(0xffffffffu, mbar_test_wait(&empty[j % S], (j / S) & 1))) {
                    issue(n_issued % S);
                    did = true;
                }
            }
            if (did) {
                idle = 0;
            } else {
                if (++idle > kWaitProbes) { failed = true; break; }
                if (idle > 32) __nanosleep(20);
            }
        }
        if (failed) {
            if (lane == 0) set_status(prm.status, TP_DEV_ERR_TIMEOUT);
            // let every issued copy land before shared memory is released
            for (int j = n_built; j < n_issued; ++j) (void)mbar_wait(&full[j % S], (j / S) & 1);
        }
    } else {
        // =========================== consumers ===========================
        const int g = warp - 1;
        const int ch0 = (g * 32 + lane) * CPT;
        float acc[RO][CPT];
#pragma unroll
        for (int r = 0; r < RO; ++r)
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;
        for (int i = 0;; ++i) {
            const int s = i % S;
            if (!__all_sync(0xffffffffu, mbar_wait(&ready[s], (i / S) & 1))) {
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_TIMEOUT);
                break;
            }
            const ChunkMeta m = meta[s];
            if (!(m.bits & kValid)) break;
            if (m.bits & kFirst) {
#pragma unroll
                for (int r = 0; r < RO; ++r)
#pragma unroll
                    for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;
            }
            const unsigned char *sb = stages + s * L.stage_bytes;
            const float *Ms = Mst + s * L.eps * P.R;
            for (int q = 0; q < m.n; ++q) {
                if (!((m.bits >> (8 + q)) & 1u)) continue;
                const FT *xs = reinterpret_cast<const FT *>(sb + L.f_off + q * L.f_bytes);
                const FT *ws = reinterpret_cast<const FT *>(sb + L.w_off + q * L.w_bytes);
                const float *Mq = Ms + q * P.R;
                float xr[RI][CPT];
#pragma unroll
                for (int l = 0; l <= LI; ++l)
#pragma unroll
                    for (int i2 = 0; i2 < 2 * l + 1; ++i2) load_vec<CPT>(xs + prm.x_off[l] + i2 * mul + ch0, xr[l * l + i2]);
                static_for<P.n>([&](auto tc) {
                    constexpr int T = decltype(tc)::value;
                    team_path<LI, LSH, LO, T, CPT, FT>(acc, xr, ws, Mq, ch0, prm.wofs[T]);
                });
            }
            if (m.bits & kLast) {
                float *orow;
                if (m.bits & kHead) orow = prm.carry + (int64_t)(2 * cta) * prm.dim_out;
                else if (m.bits & kTail) orow = prm.carry + (int64_t)(2 * cta + 1) * prm.dim_out;
                else orow = prm.out + (int64_t)m.seg * prm.dim_out;
#pragma unroll
                for (int l = 0; l <= LO; ++l) {
                    const int off = prm.o_off[l];
                    if (off < 0) continue;
#pragma unroll
                    for (int k = 0; k < 2 * l + 1; ++k) store_vec<CPT>(orow + off + k * mul + ch0, acc[l * l + k]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
}

// out[d] = tail partial of the stream where d starts + head partials of the
// following streams that continue d, added in stream order. One warp per stream.
__global__ void carry_fixup_kernel(const float *__restrict__ carry, const int32_t *__restrict__ carry_dst, int n_streams,
                                   int dim_out, float *__restrict__ out);

}  // namespace tpc
