// Forward kernel for irreps shapes with a compile-time path program
// (program.h) in the natural layout (input blocks l = 0..LI, output blocks
// l = 0..LO, mul = 32*CPT channels each, paths in program order): every warp
// warp is an independent pipeline that copies its own edges into a private
// S-stage shared-memory ring with 1-D bulk (TMA) copies and consumes them
// itself. There is no producer warp and no barrier between warps; the only
// synchronisation is the warp's own mbarrier per stage.
//
// Work split: the destination-sorted edge list is cut into `n_pieces` exact,
// contiguous, equal pieces; piece p belongs to warp p % n_warps, so with
// several pieces per warp ("rounds") the whole grid sweeps the edge list front
// to back together, which keeps the gathered source rows of neighbouring
// destinations in L2 at the same time.
//
// Per warp:
//   issue:   chunks of up to `eps` consecutive edges of its pieces, in order;
//            one bulk copy for the chunk's weight rows, one for the 16-byte
//            aligned span around its harmonic rows (each from its own lane),
//            and the gathered source rows x[src[e]] by 16-byte cp.async, every
//            lane a 16-byte slice of each row. The source indices of the
//            next two chunks are loaded ahead into registers; an out-of-range
//            source sets a status bit and its edge gets a zero row.
//   consume: wait for the chunk's stage, build the per-edge matrices
//            M_p[i][k] = sum_j C_p[i,j,k] sh[j] (program layout, at most two
//            terms per entry) into a warp-private buffer, then run every path as
//            straight-line code into the destination row held in registers
//            (lane = CPT consecutive channels, so one warp covers all channels;
//            with PK two channels share one packed fma.rn.f32x2, whose halves
//            round exactly like two fmaf: half the issue slots, but a longer
//            dependent latency), refill the stage with the chunk S ahead.
//   store:   when a destination ends its row is written once; a destination cut
//            by a piece boundary is written as a head/tail partial that
//            carry_fixup_kernel adds in piece order. No atomics: results are
//            bitwise reproducible for a given launch geometry.
#pragma once
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "conv_common.cuh"
#include "program.h"
#include "tuning.h"

namespace tpc {

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

// out[d] = tail partial of the piece where d starts + head partials of the
// following pieces that continue d, added in piece order. One warp per piece.
// Destination ids outside [0, n_dst) (a piece a failed warp never reached
// holds -1) are skipped.
__global__ void carry_fixup_kernel(const float *__restrict__ carry, const int32_t *__restrict__ carry_dst, int n_pieces,
                                   int dim_out, int n_dst, float *__restrict__ out);


// Width of the radial network's hidden layer (Linear(1, 16) -> SiLU -> Linear(16, P*mul)).
constexpr int kMlpHidden = 16;

// The radial network with edge pairs (one channel per lane, at most
// kMlpMaxPaths paths) forms the weights in registers, two edges per packed
// FMA: the block keeps a copy of the second layer arranged by lane,
// [i][half][lane][4] = w2[i][4*half .. 4*half+3][c] (zero past the last path;
// i = kMlpHidden holds the bias), and a chunk of at most kMlpChunk edges reads
// that copy once and gets its weights, paired by edge, by 16 packed FMAs each
// (the value splatted into both halves in registers). kMlpSplat keeps the
// splatted pairs in shared memory instead, [i][j][lane][4] = {w2[i][2j][c]
// twice, w2[i][2j+1][c] twice}: no register moves, but twice the
// shared-memory reads, which measured 5 % slower.
constexpr int kMlpChunk = 8, kMlpMaxPaths = 8;
constexpr bool kMlpSplat = false;
constexpr int kMlpW2sBytes = (kMlpHidden + 1) * (kMlpSplat ? 4 : 2) * 32 * 16;

struct RingParams {
    int32_t S, eps;                      // stages per warp, edges per chunk (<= 30)
    int32_t stage_bytes, f_off, sh_off;  // stage: weight rows at 0 (none in VM 2's own layouts), source rows, harmonic span
    int32_t m_off, bar_off, warp_bytes;  // warp region: stages, M, barriers
    int32_t y_off;                       // warp region: harmonics computed from edge vectors [eps][SHN]
    int32_t vec_mode;                    // kernels with VM >= 1: 1 harmonics of the unit vector, 2 raw polynomial
    int32_t h_off;                       // warp region (VM == 2): hidden activations, [eps][kMlpHidden]
                                         // (edge pairs: [kMlpHidden][kMlpChunk], then kMlpChunk lengths)
    const float *mlp_w1, *mlp_b1;        // VM == 2: [H], [H]
    const float *mlp_w2, *mlp_b2;        // VM == 2: [H][P*mul] (h-major), [P*mul]
    int32_t tab_bytes;                   // block-shared bytes: the M recipe table, then (VM 2, edge pairs)
    int32_t w2s_off;                     // the second layer's copy by lane
    uint32_t ej[kMaxM];
    float ec[kMaxM][2];
    const void *x;
    const float *sh;
    const void *w;
    const int32_t *src;
    const int32_t *row_ptr;
    float *out;
    float *carry;        // [2*n_pieces][dim_out]
    int32_t *carry_dst;  // [2*n_pieces]
    int *status;
    int32_t n_src, n_dst, n_warps, n_pieces;
    int64_t E;
    uint64_t wait_ns;    // main-loop pipeline wait limit
};

// Smallest d in [0, N] with rp[d] >= target (N+1 if none): one lane's binary search.
__device__ __forceinline__ int lane_first_geq(const int32_t *rp, int N, int64_t target) {
    int lo = 0, hi = N + 1;
    while (lo < hi) {
        const int mid = lo + ((hi - lo) >> 1);
        if ((int64_t)rp[mid] >= target) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// ---- lane values: CPT channels as floats (CPT = 1) or packed pairs (CPT >= 2) ----
typedef unsigned long long f32x2;

__device__ __forceinline__ void vfma(float &d, float a, float b) { d = fmaf(a, b, d); }
__device__ __forceinline__ float vmul(float a, float b) { return a * b; }
__device__ __forceinline__ void vfma(f32x2 &d, f32x2 a, f32x2 b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ f32x2 vmul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float lo_f(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }

// PK with CPT >= 2: a lane value is two neighbouring channels of one edge.
// PK with CPT == 1 ("edge pairs"): a lane value is one channel of two
// consecutive edges of the same destination, whose partial sums are kept
// apart and added when the destination is stored.
template <int CPT, bool PK>
struct LaneVec {
    static constexpr bool kPair = PK;
    static constexpr bool kEdgePair = PK && CPT == 1;
    static constexpr int NV = kPair ? (kEdgePair ? 1 : CPT / 2) : CPT;
    using V = typename std::conditional<kPair, f32x2, float>::type;
};

// CPT consecutive channels starting at p (shared memory), as lane values.
template <int CPT, bool PK>
__device__ __forceinline__ void load_lane(const float *p, typename LaneVec<CPT, PK>::V (&v)[LaneVec<CPT, PK>::NV]) {
    if constexpr (LaneVec<CPT, PK>::kPair) {
        if constexpr (CPT == 4) {
            const ulonglong2 t = *reinterpret_cast<const ulonglong2 *>(p);
            v[0] = t.x;
            v[1] = t.y;
        } else {
            v[0] = *reinterpret_cast<const f32x2 *>(p);
        }
    } else {
        load_vec<CPT>(p, v);
    }
}
template <int CPT, bool PK>
__device__ __forceinline__ void load_lane(const __nv_bfloat16 *p,
                                          typename LaneVec<CPT, PK>::V (&v)[LaneVec<CPT, PK>::NV]) {
    if constexpr (LaneVec<CPT, PK>::kPair) {
        if constexpr (CPT == 4) {
            const uint2 t = *reinterpret_cast<const uint2 *>(p);
            v[0] = pack2(bf16lo(t.x), bf16hi(t.x));
            v[1] = pack2(bf16lo(t.y), bf16hi(t.y));
        } else {
            const uint32_t t = *reinterpret_cast<const uint32_t *>(p);
            v[0] = pack2(bf16lo(t), bf16hi(t));
        }
    } else {
        load_vec<CPT>(p, v);
    }
}

// Does entry q of path T write an accumulator row k that no earlier entry wrote?
template <int LI, int LSH, int LO>
constexpr bool first_of_k(int T, int q) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    for (int q2 = 0; q2 < q; ++q2)
        if ((P.ik[T][q2] & 7) == (P.ik[T][q] & 7)) return false;
    return true;
}
template <int LI, int LSH, int LO>
constexpr bool has_k(int T, int k) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    for (int q = 0; q < P.nz[T]; ++q)
        if ((P.ik[T][q] & 7) == k) return true;
    return false;
}
template <int LI, int LSH, int LO>
constexpr bool has_i(int T, int i) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    for (int q = 0; q < P.nz[T]; ++q)
        if ((P.ik[T][q] >> 3) == i) return true;
    return false;
}

// Emission order of the entries of path T: by rank among the entries of the
// same accumulator row k, then by position. Consecutive FMAs then mostly
// target different rows, while each row still receives its terms in program
// order (so the sums are the same as in plain order).
template <int LI, int LSH, int LO>
constexpr int entry_at(int T, int pos) {
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    int seen = 0;
    for (int rank = 0; rank < kProgMaxNz; ++rank)
        for (int q = 0; q < P.nz[T]; ++q) {
            int r = 0;
            for (int q2 = 0; q2 < q; ++q2) r += (P.ik[T][q2] & 7) == (P.ik[T][q] & 7);
            if (r != rank) continue;
            if (seen == pos) return q;
            ++seen;
        }
    return -1;
}

// One program path for one edge: acc[lc-block row k] += w_T * sum_i M_T[i][k] x[la-block row i],
// with this lane's weight values wv of the path given. Mq: the edge's M
// (entries duplicated into pairs for channel pairs, the two edges' entries
// interleaved for edge pairs).
template <int LI, int LSH, int LO, int T, int CPT, bool PK>
__device__ __forceinline__ void ring_path_w(typename LaneVec<CPT, PK>::V (&acc)[rows_upto(LO)][LaneVec<CPT, PK>::NV],
                                            const typename LaneVec<CPT, PK>::V (&xr)[rows_upto(LI)][LaneVec<CPT, PK>::NV],
                                            const typename LaneVec<CPT, PK>::V (&wv)[LaneVec<CPT, PK>::NV],
                                            const float *Mq) {
    using LV = LaneVec<CPT, PK>;
    using V = typename LV::V;
    constexpr int NV = LV::NV;
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int LA = P.p[T].la, LC = P.p[T].lc;
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NZ = P.nz[T], MO = P.moff[T];
    // M entries of this path: 4 per 16-byte load (singles) or 2 (pairs)
    constexpr int PER = LV::kPair ? 2 : 4;
    constexpr int NL = (NZ + PER - 1) / PER;
    V m[NL * PER];
    if constexpr (LV::kPair) {
        const ulonglong2 *M2 = reinterpret_cast<const ulonglong2 *>(Mq + 2 * MO);
#pragma unroll
        for (int q = 0; q < NL; ++q) {
            const ulonglong2 t = M2[q];
            m[2 * q] = t.x;
            m[2 * q + 1] = t.y;
        }
    } else {
        const float4 *M4 = reinterpret_cast<const float4 *>(Mq + MO);
#pragma unroll
        for (int q = 0; q < NL; ++q) {
            const float4 t = M4[q];
            m[4 * q] = t.x;
            m[4 * q + 1] = t.y;
            m[4 * q + 2] = t.z;
            m[4 * q + 3] = t.w;
        }
    }
    if constexpr (NA <= NC) {
        V wx[NA][NV];
        static_for<NA>([&](auto ic) {
            constexpr int i = decltype(ic)::value;
            if constexpr (has_i<LI, LSH, LO>(T, i)) {
#pragma unroll
                for (int c = 0; c < NV; ++c) wx[i][c] = vmul(wv[c], xr[LA * LA + i][c]);
            }
        });
        static_for<NZ>([&](auto pc) {
            constexpr int q = entry_at<LI, LSH, LO>(T, decltype(pc)::value);
            constexpr int i = P.ik[T][q] >> 3, k = P.ik[T][q] & 7;
#pragma unroll
            for (int c = 0; c < NV; ++c) vfma(acc[LC * LC + k][c], m[q], wx[i][c]);
        });
    } else {
        V tk[NC][NV];
        static_for<NZ>([&](auto pc) {
            constexpr int q = entry_at<LI, LSH, LO>(T, decltype(pc)::value);
            constexpr int i = P.ik[T][q] >> 3, k = P.ik[T][q] & 7;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                if constexpr (first_of_k<LI, LSH, LO>(T, q)) tk[k][c] = vmul(m[q], xr[LA * LA + i][c]);
                else vfma(tk[k][c], m[q], xr[LA * LA + i][c]);
            }
        });
        static_for<NC>([&](auto kc) {
            constexpr int k = decltype(kc)::value;
            if constexpr (has_k<LI, LSH, LO>(T, k)) {
#pragma unroll
                for (int c = 0; c < NV; ++c) vfma(acc[LC * LC + k][c], wv[c], tk[k][c]);
            }
        });
    }
}

// The same with the weights read from shared memory. wl: this lane's channels
// of the edge's weight row (wlB: of the second edge, edge pairs only); use_a /
// use_b: edge pairs only, whether each edge takes part (an absent one adds zero).
template <int LI, int LSH, int LO, int T, int CPT, bool PK, typename FT>
__device__ __forceinline__ void ring_path(typename LaneVec<CPT, PK>::V (&acc)[rows_upto(LO)][LaneVec<CPT, PK>::NV],
                                          const typename LaneVec<CPT, PK>::V (&xr)[rows_upto(LI)][LaneVec<CPT, PK>::NV],
                                          const FT *wl, const FT *wlB, const float *Mq, bool use_a = true,
                                          bool use_b = true) {
    using LV = LaneVec<CPT, PK>;
    constexpr int MUL = 32 * CPT;
    typename LV::V wv[LV::NV];
    if constexpr (LV::kEdgePair) {
        const float a = to_float(wl[T * MUL]), b = to_float(wlB[T * MUL]);
        wv[0] = pack2(use_a ? a : 0.f, use_b ? b : 0.f);
    } else {
        load_lane<CPT, PK>(wl + T * MUL, wv);
    }
    ring_path_w<LI, LSH, LO, T, CPT, PK>(acc, xr, wv, Mq);
}

// CPT consecutive floats of read-only global memory (4*CPT-byte aligned).
template <int CPT>
__device__ __forceinline__ void ldg_lane(const float *p, float (&v)[CPT]) {
    if constexpr (CPT == 4) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = t.x;
        v[1] = t.y;
        v[2] = t.z;
        v[3] = t.w;
    } else if constexpr (CPT == 2) {
        const float2 t = __ldg(reinterpret_cast<const float2 *>(p));
        v[0] = t.x;
        v[1] = t.y;
    } else {
        v[0] = __ldg(p);
    }
}

template <int CPT, bool PK>
__device__ __forceinline__ void store_lane(float *p, const typename LaneVec<CPT, PK>::V (&v)[LaneVec<CPT, PK>::NV]) {
    if constexpr (LaneVec<CPT, PK>::kEdgePair) *p = lo_f(v[0]) + hi_f(v[0]);
    else if constexpr (!LaneVec<CPT, PK>::kPair) store_vec<CPT>(p, v);
    else if constexpr (CPT == 4) *reinterpret_cast<ulonglong2 *>(p) = make_ulonglong2(v[0], v[1]);
    else *reinterpret_cast<f32x2 *>(p) = v[0];
}

// Does the launch's shared-memory layout (RingParams offsets, dynamic size)
// hold every region ring_fwd_kernel<...> writes? Kept out of line so the
// kernel's own register allocation does not carry it.
template <int LI, int LSH, int LO, int CPT, bool PK, typename FT, int VM>
__device__ __noinline__ bool ring_layout_ok(const RingParams &prm, int warps_per_block) {
    using LV = LaneVec<CPT, PK>;
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int MUL = 32 * CPT, SHN = rows_upto(LSH);
    constexpr int WB = P.n * MUL * (int)sizeof(FT), FB = rows_upto(LI) * MUL * (int)sizeof(FT);
    constexpr int MS = LV::kPair ? 2 * P.R : P.R;
    constexpr int HR = VM >= 1 ? 3 : SHN;
    constexpr bool pair_mlp = VM == 2 && LV::kEdgePair && P.n <= kMlpMaxPaths;
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const int e = prm.eps;
    return e >= 1 && e <= (pair_mlp ? kMlpChunk : 30) && prm.S >= 1 &&
           ((prm.f_off | prm.sh_off | prm.stage_bytes | prm.m_off | prm.y_off | prm.h_off | prm.bar_off |
             prm.warp_bytes | prm.tab_bytes) & 15) == 0 &&
           prm.tab_bytes >= 16 * P.R &&
           (!pair_mlp || (prm.w2s_off >= 16 * P.R && prm.w2s_off + kMlpW2sBytes <= prm.tab_bytes)) &&
           prm.f_off >= (VM == 2 ? 0 : e * WB) && prm.sh_off >= prm.f_off + e * FB &&
           prm.stage_bytes >= prm.sh_off + e * HR * 4 + (HR % 4 ? 32 : 0) && prm.m_off >= prm.S * prm.stage_bytes &&
           prm.y_off >= prm.m_off + e * MS * 4 && (VM == 0 || prm.h_off >= prm.y_off + e * SHN * 4) &&
           (VM != 2 || prm.bar_off >= prm.h_off + (pair_mlp ? kMlpChunk * (kMlpHidden + 1) : e * kMlpHidden) * 4) &&
           prm.warp_bytes >= prm.bar_off + prm.S * 8 &&
           (int64_t)prm.tab_bytes + (int64_t)warps_per_block * prm.warp_bytes <= (int64_t)dyn;
}

// CPT channels per lane (mul = 32*CPT), PK: packed pairs of channels. The
// register cap follows from MINB (blocks of 256 threads per SM). VM (vector
// mode) 0: `sh` holds harmonic rows; 1: `sh` holds edge vectors [E][3] and the
// harmonics are evaluated here; 2: as 1, and the weights are computed here
// too, by the radial network Linear(1,H) -> SiLU -> Linear(H,P*mul) of the edge
// length, instead of streamed from `w`: with edge pairs a chunk's at once in
// registers, with plain lanes or channel pairs each path's right before the
// path, else (edge pairs of the larger programs) as weight rows in the stage.
template <int LI, int LSH, int LO, int CPT, bool PK, int MINB, typename FT, int VM>
__global__ void __launch_bounds__(32 * kRingMaxWarps, MINB) ring_fwd_kernel(const __grid_constant__ RingParams prm) {
    using LV = LaneVec<CPT, PK>;
    using V = typename LV::V;
    constexpr int NV = LV::NV;
    constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    constexpr int RI = rows_upto(LI), RO = rows_upto(LO);
    constexpr int KR = (P.R + 31) / 32;
    constexpr int MUL = 32 * CPT;
    constexpr int DX = RI * MUL, DOUT = RO * MUL, SHN = rows_upto(LSH);
    constexpr int WNUM = P.n * MUL;
    constexpr int WB = WNUM * (int)sizeof(FT), FB = DX * (int)sizeof(FT);
    constexpr int MS = LV::kPair ? 2 * P.R : P.R;  // M floats per edge
    static_assert(WB % 16 == 0 && FB % 16 == 0, "bulk copies move 16-byte multiples");
    extern __shared__ __align__(128) unsigned char smem[];
    static_assert(MS % 4 == 0, "M rows are read with 16-byte loads");
    // the launch's layout must hold everything this instantiation writes:
    // checked before the first shared-memory store, a mismatch (a library
    // bug) is reported and nothing runs
    if (!ring_layout_ok<LI, LSH, LO, CPT, PK, FT, VM>(prm, blockDim.x >> 5)) {
        if (threadIdx.x == 0) set_status(prm.status, TP_DEV_ERR_INTERNAL);
        return;
    }
    // block-shared recipe of the M entries: r -> {4*j0, 4*j1, c0, c1},
    // M[r] = c0 * sh[j0] + c1 * sh[j1]
    int4 *tab = reinterpret_cast<int4 *>(smem);
    for (int r = threadIdx.x; r < P.R; r += blockDim.x)
        tab[r] = make_int4((int)(prm.ej[r] & 0xffffu) * 4, (int)(prm.ej[r] >> 16) * 4, __float_as_int(prm.ec[r][0]),
                           __float_as_int(prm.ec[r][1]));
    // radial network with edge pairs: weights formed in registers from a block copy of the second layer
    constexpr bool kMlpReg = VM == 2 && LV::kEdgePair && P.n <= kMlpMaxPaths;
    // radial network with plain lanes or channel pairs: each path's weights
    // formed in registers just before the path, from 16-byte loads of the
    // lane's channels of w2 and b2
    constexpr bool kMlpCols = VM == 2 && !LV::kEdgePair;
    if constexpr (kMlpReg) {
        float *w2s = reinterpret_cast<float *>(smem + prm.w2s_off);
        for (int t = threadIdx.x; t < kMlpW2sBytes / 4; t += blockDim.x) {
            const int i = kMlpSplat ? t >> 9 : t >> 8, c = (t >> 2) & 31;
            const int p = kMlpSplat ? 2 * ((t >> 7) & 3) + ((t >> 1) & 1) : 4 * ((t >> 7) & 1) + (t & 3);
            float v = 0.f;
            if (p < P.n) v = i < kMlpHidden ? prm.mlp_w2[i * WNUM + p * MUL + c] : prm.mlp_b2[p * MUL + c];
            w2s[t] = v;
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int gw = blockIdx.x * (blockDim.x >> 5) + wib;
    if (gw >= prm.n_warps) return;
    const int S = prm.S, eps = prm.eps;
    unsigned char *base = smem + prm.tab_bytes + (size_t)wib * prm.warp_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + prm.bar_off);
    float *Mw = reinterpret_cast<float *>(base + prm.m_off);
    // kXAsync: source rows by 16-byte cp.async per lane (the load/store unit)
    // instead of one bulk copy per row (measured 1-3 % faster on every program
    // shape); the stage's barrier then also takes one arrival per lane, when
    // that lane's copies have landed
    constexpr bool kXAsync = true;
    if (lane == 0)
        for (int s = 0; s < S; ++s) mbar_init(&full[s], kXAsync ? 33 : 1);
    fence_barrier_init();
    if constexpr (LV::kEdgePair)  // an absent second edge reads finite (zero) M entries
        for (int i = lane; i < eps * MS; i += 32) Mw[i] = 0.f;
    __syncwarp();

    const int nP = prm.n_pieces, nW = prm.n_warps, N = prm.n_dst;
    const int E = (int)prm.E;  // the host launches this kernel only for E < 2^31
    const int32_t *rp = prm.row_ptr;
    const int32_t *srcp = prm.src;
    const FT *xp = static_cast<const FT *>(prm.x);
    const unsigned char *wb = static_cast<const unsigned char *>(prm.w);
    const unsigned char *shb_g = reinterpret_cast<const unsigned char *>(prm.sh);
    const int ch0 = lane * CPT;
    auto piece_lo = [&](int p) -> int { return (int)((int64_t)p * E / nP); };

    // ---- issue side: chunk cursors over this warp's pieces -------------------------
    // A chunk is the next min(eps, hi - e) edges of the current piece; the
    // consumer walks the same sequence, so nothing about a chunk but its data
    // goes through shared memory.
    struct Cur {
        int p, e, hi, n;
    };
    auto settle = [&](Cur &c) {  // skip finished pieces, then size the chunk
        while (c.p < nP && c.e >= c.hi) {
            c.p += nW;
            if (c.p < nP) {
                c.e = piece_lo(c.p);
                c.hi = piece_lo(c.p + 1);
            }
        }
        c.n = c.p < nP ? min(eps, c.hi - c.e) : 0;
    };
    auto load_src = [&](const Cur &c) -> int { return lane < c.n ? srcp[c.e + lane] : -1; };
    Cur ic{gw, gw < nP ? piece_lo(gw) : 0, gw < nP ? piece_lo(gw + 1) : 0, 0};
    settle(ic);
    Cur lc = ic;  // one chunk ahead of ic
    lc.e += lc.n;
    settle(lc);
    int srcA = load_src(ic), srcB = load_src(lc);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    // the streamed per-edge rows: harmonics (SHN floats) or edge vectors (3 floats)
    constexpr bool VEC = VM >= 1;
    static_assert(VM != 2 || sizeof(FT) == 4, "computed weight rows are float32");
    constexpr int HR = VEC ? 3 : SHN;
    const int64_t sh_bytes_all = (int64_t)E * HR * 4;
    int n_issued = 0, s_iss = 0;
    auto issue_next = [&]() {
        const int n = ic.n;
        if (n == 0) return;
        const int s = s_iss;
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        unsigned char *sb = base + s * prm.stage_bytes;
        const bool ok = (uint32_t)srcA < (uint32_t)prm.n_src;
        const uint32_t okmask = __ballot_sync(0xffffffffu, ok) & (n == 32 ? 0xffffffffu : (1u << n) - 1u);
        // harmonic rows [e, e+n): one bulk copy of the 16-byte aligned span around
        // them; a piece past the array's last 16-byte boundary by plain loads
        const int64_t b0 = (int64_t)ic.e * HR * 4, b1 = (int64_t)(ic.e + n) * HR * 4;
        int64_t a0 = b0, a1 = b1;  // rows of a multiple of 4 floats: the span is aligned already
        if constexpr (HR % 4 != 0) {
            a0 = b0 & ~(int64_t)15;
            a1 = (b1 + 15) & ~(int64_t)15;
            if (a1 > sh_bytes_all) a1 = sh_bytes_all & ~(int64_t)15;
            if (a1 < a0) a1 = a0;
            if (a1 < b1) {
                const float *sf = prm.sh + a1 / 4;
                float *df = reinterpret_cast<float *>(sb + prm.sh_off) + (a1 - a0) / 4;
                for (int q = lane; q < (int)((b1 - a1) / 4); q += 32) df[q] = sf[q];
            }
        }
        const uint32_t sh_tma = (uint32_t)(a1 - a0);
        if (okmask != (n == 32 ? 0xffffffffu : (1u << n) - 1u)) {
            // an edge with an out-of-range source: flag it, and give it a zero row
            if (lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
            for (int q = 0; q < n; ++q)
                if (!((okmask >> q) & 1u))
                    for (int o = lane * 16; o < FB; o += 512)
                        *reinterpret_cast<uint4 *>(sb + prm.f_off + q * FB + o) = make_uint4(0, 0, 0, 0);
        }
        const uint32_t w_tma = VM == 2 ? 0u : (uint32_t)n * WB;  // VM 2: weight rows computed, not copied
        const uint32_t x_tma = kXAsync ? 0u : (uint32_t)__popc(okmask) * FB;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], w_tma + x_tma + sh_tma);
        if constexpr (kXAsync) {
            const unsigned char *xg = reinterpret_cast<const unsigned char *>(xp);
            for (int q = 0; q < n; ++q) {  // warp-uniform: every lane takes part in every shuffle
                const int sq = __shfl_sync(0xffffffffu, srcA, q);
                if ((okmask >> q) & 1u) {
                    const unsigned char *g = xg + (int64_t)sq * FB;
                    unsigned char *d = sb + prm.f_off + q * FB;
#pragma unroll
                    for (int o = lane * 16; o < FB; o += 512) cp_async16(d + o, g + o);
                }
            }
            cp_async_mbar_arrive_noinc(&full[s]);
        }
        __syncwarp();
        // one bulk copy per lane: lane 0 the weight rows, lane 1 the harmonic
        // span, and (kXAsync false) lane 2 + q the source row of edge q
        const int xs = __shfl_up_sync(0xffffffffu, srcA, 2);
        const int q = lane - 2;
        const void *gsrc = wb + (int64_t)ic.e * WB;
        unsigned char *sdst = sb;
        uint32_t nbytes = w_tma;
        uint64_t pol = pol_stream;
        if (lane == 1) {
            gsrc = shb_g + a0;
            sdst = sb + prm.sh_off;
            nbytes = sh_tma;
        } else if (lane >= 2) {
            gsrc = xp + (int64_t)xs * DX;
            sdst = sb + prm.f_off + q * FB;
            nbytes = (!kXAsync && q < n && ((okmask >> q) & 1u)) ? (uint32_t)FB : 0u;
            pol = pol_keep;
        }
        if (nbytes) bulk_g2s(sdst, gsrc, nbytes, &full[s], pol);
        // the source indices a few chunks on start their way to L2 now, so the
        // register load two chunks ahead does not wait on HBM
        if (lane == 0 && ic.e + 16 * eps < E) asm volatile("prefetch.global.L2 [%0];" ::"l"(srcp + ic.e + 16 * eps));
        ++n_issued;
        ic = lc;
        srcA = srcB;
        lc.e += lc.n;
        settle(lc);
        srcB = load_src(lc);
    };
    for (int k = 0; k < S; ++k) issue_next();

    // ---- destination ranges of this warp's pieces -------------------------------
    // F(e) = smallest d with row_ptr[d] >= e. Piece p covers destinations
    // [F(lo(p)) (-1 if that one starts before lo(p)), F(lo(p+1))), the last piece up to N.
    const int np_w = gw < nP ? (nP - 1 - gw) / nW + 1 : 0;
    int fb = 0;  // lane i < 2*np_w: F(lo(p_{i/2} + (i&1)))
    if (np_w == 1) {
        const int f0 = warp_first_geq(rp, N, piece_lo(gw), lane);
        const int f1 = warp_first_geq(rp, N, piece_lo(gw + 1), lane);
        fb = lane == 0 ? f0 : f1;
    } else if (lane < 2 * np_w) {
        fb = lane_first_geq(rp, N, piece_lo(gw + (lane >> 1) * nW + (lane & 1)));
    }
    // and row_ptr there, so a piece starts without a dependent load
    const int rb = lane < 2 * np_w ? rp[min(fb, N)] : 0;
    auto piece_dstart = [&](int j) {  // first destination of piece j and whether it began earlier
        const int e_lo = piece_lo(gw + j * nW);
        int d = min(__shfl_sync(0xffffffffu, fb, 2 * j), N);
        const bool earlier = d > 0 && __shfl_sync(0xffffffffu, rb, 2 * j) > e_lo;
        return earlier ? -(d - 1) - 1 : d;  // negative: d-1 started in an earlier piece
    };
    // row_ptr window of the next piece, loaded one piece ahead
    int wv_next = 0, wbase_next = -1;
    auto prefetch_window = [&](int j) {
        if (j >= np_w) return;
        const int ds = piece_dstart(j);
        wbase_next = ds < 0 ? -ds - 1 : ds;
        wv_next = (wbase_next + lane <= N) ? rp[wbase_next + lane] : 0;
    };
    prefetch_window(0);

    // ---- consume side ---------------------------------------------------------------
    V acc[RO][NV];
#pragma unroll
    for (int r = 0; r < RO; ++r)
#pragma unroll
        for (int c = 0; c < NV; ++c) acc[r][c] = V(0);
    int n_done = 0, s_done = 0;
    uint32_t ph_done = 0;
    bool failed = false;
    int failed_j = 0;  // the piece whose wait gave up
    for (int j = 0; j < np_w && !failed; ++j) {
        const int p = gw + j * nW;
        const int e_lo = piece_lo(p), e_hi = piece_lo(p + 1);
        const int ds = piece_dstart(j);
        const int d_start = ds < 0 ? -ds - 1 : ds;
        int d_end = __shfl_sync(0xffffffffu, fb, 2 * j + 1);
        const int rp_end = __shfl_sync(0xffffffffu, rb, 2 * j + 1);  // row_ptr[min(d_end, N)]
        if (p == nP - 1 || d_end > N) d_end = N;
        if (d_end < d_start) d_end = d_start;
        // d_start began in an earlier piece: a head partial; d_end - 1 runs on past e_hi: a tail partial
        const int head_dst = (ds < 0 && d_start < d_end) ? d_start : -1;
        int tail_dst = (p < nP - 1 && d_end > d_start && rp_end > e_hi) ? d_end - 1 : -1;
        if (tail_dst == head_dst) tail_dst = -1;
        if (lane == 0) {
            prm.carry_dst[2 * p] = head_dst;
            prm.carry_dst[2 * p + 1] = tail_dst;
        }
        // row_ptr window: lane l holds rp[wbase + l]
        int wbase = wbase_next;
        int32_t wv = wv_next;
        prefetch_window(j + 1);
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
        };
        auto store_row = [&](int d) {
            float *orow;
            if (d == head_dst) orow = prm.carry + (int64_t)(2 * p) * DOUT;
            else if (d == tail_dst) orow = prm.carry + (int64_t)(2 * p + 1) * DOUT;
            else orow = prm.out + (int64_t)d * DOUT;
            orow += ch0;
#pragma unroll
            for (int r = 0; r < RO; ++r) store_lane<CPT, PK>(orow + r * MUL, acc[r]);
#pragma unroll
            for (int r = 0; r < RO; ++r)
#pragma unroll
                for (int c = 0; c < NV; ++c) acc[r][c] = V(0);
        };
        enter(cur_d);
        int e = e_lo;
        while (e < e_hi) {
            const int s = s_done;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph_done, prm.wait_ns))) {
                failed = true;  // reported, and its pieces marked, after the loop
                failed_j = j;
                break;
            }
            const int n = min(eps, e_hi - e);
            const unsigned char *sb = base + s * prm.stage_bytes;
            if constexpr (kMlpReg) {
                // harmonics of the chunk's edge vectors and their lengths (one
                // edge per lane), then the hidden activations h[i][q], q < kMlpChunk
                // (zero-length past n), each lane one q and four i
                const float *vq = reinterpret_cast<const float *>(sb + prm.sh_off + (e * HR & 3) * 4);
                float *Y = reinterpret_cast<float *>(base + prm.y_off);
                float *hq = reinterpret_cast<float *>(base + prm.h_off);
                float *rq = hq + kMlpChunk * kMlpHidden;
                if (lane < kMlpChunk) {
                    float r = 0.f;
                    if (lane < n) {
                        const float vx = vq[3 * lane], vy = vq[3 * lane + 1], vz = vq[3 * lane + 2];
                        float yv[16];
                        real_sh_upto<LSH>(vx, vy, vz, prm.vec_mode == 1, yv);
#pragma unroll
                        for (int j = 0; j < SHN; ++j) Y[lane * SHN + j] = yv[j];
                        r = sqrtf(vx * vx + vy * vy + vz * vz);
                    }
                    rq[lane] = r;
                }
                __syncwarp();
                const float r = rq[lane & (kMlpChunk - 1)];
#pragma unroll
                for (int k = 0; k < kMlpHidden * kMlpChunk / 32; ++k) {
                    const int i = (lane >> 3) + 4 * k;
                    const float z = fmaf(__ldg(prm.mlp_w1 + i), r, __ldg(prm.mlp_b1 + i));
                    hq[i * kMlpChunk + (lane & (kMlpChunk - 1))] = __fdividef(z, 1.f + __expf(-z));
                }
            } else if constexpr (VM == 2) {
                // weight rows of the chunk from the radial network of the edge length:
                // h[q][i] = silu(w1[i] |v_q| + b1[i]), w[q][j] = b2[j] + sum_i w2[i][j] h[q][i]
                const float *vq = reinterpret_cast<const float *>(sb + prm.sh_off + (e * HR & 3) * 4);
                float *hq = reinterpret_cast<float *>(base + prm.h_off);
                constexpr int H = kMlpHidden;
                for (int t = lane; t < n * H; t += 32) {
                    const int q = t / H, i = t - q * H;
                    const float vx = vq[3 * q], vy = vq[3 * q + 1], vz = vq[3 * q + 2];
                    const float r = sqrtf(vx * vx + vy * vy + vz * vz);
                    const float z = fmaf(__ldg(prm.mlp_w1 + i), r, __ldg(prm.mlp_b1 + i));
                    hq[q * H + i] = z / (1.f + expf(-z));
                }
                __syncwarp();
            }
            if constexpr (VM == 2 && !kMlpReg && !kMlpCols) {
                constexpr int H = kMlpHidden;
                const float *hq = reinterpret_cast<const float *>(base + prm.h_off);
                float *wrows = reinterpret_cast<float *>(const_cast<unsigned char *>(sb));
                // U columns per lane at a time: U independent 16-FMA chains (and
                // their 16*U loads in flight) instead of one, where the register
                // budget allows (one block per SM); each column's sum keeps its order
                constexpr int U = MINB == 1 ? 8 : 1;
                auto columns = [&](int j, auto uc) {
                    constexpr int NU = decltype(uc)::value;
                    float w2c[NU][H], bj[NU];
#pragma unroll
                    for (int u = 0; u < NU; ++u) {
#pragma unroll
                        for (int i = 0; i < H; ++i) w2c[u][i] = __ldg(prm.mlp_w2 + i * WNUM + j + 32 * u);
                        bj[u] = __ldg(prm.mlp_b2 + j + 32 * u);
                    }
                    for (int q = 0; q < n; ++q) {
                        const float4 *h4 = reinterpret_cast<const float4 *>(hq + q * H);
                        float a[NU];
#pragma unroll
                        for (int u = 0; u < NU; ++u) a[u] = bj[u];
#pragma unroll
                        for (int i4 = 0; i4 < H / 4; ++i4) {
                            const float4 hv = h4[i4];
#pragma unroll
                            for (int u = 0; u < NU; ++u) {
                                a[u] = fmaf(w2c[u][4 * i4], hv.x, a[u]);
                                a[u] = fmaf(w2c[u][4 * i4 + 1], hv.y, a[u]);
                                a[u] = fmaf(w2c[u][4 * i4 + 2], hv.z, a[u]);
                                a[u] = fmaf(w2c[u][4 * i4 + 3], hv.w, a[u]);
                            }
                        }
#pragma unroll
                        for (int u = 0; u < NU; ++u) wrows[q * WNUM + j + 32 * u] = a[u];
                    }
                };
                int j = lane;
                for (; j + 32 * (U - 1) < WNUM; j += 32 * U) columns(j, std::integral_constant<int, U>{});
                for (; j < WNUM; j += 32) columns(j, std::integral_constant<int, 1>{});
                __syncwarp();
            }
            // M of the chunk's edges (lane-parallel over entries)
            {
                const unsigned char *shq = sb + prm.sh_off + (HR % 4 != 0 ? (e * HR & 3) * 4 : 0);
                if constexpr (kMlpReg) {
                    shq = reinterpret_cast<const unsigned char *>(base + prm.y_off);  // evaluated above
                } else if constexpr (VEC) {
                    // harmonics of the chunk's edge vectors, one edge per lane
                    float *Y = reinterpret_cast<float *>(base + prm.y_off);
                    if (lane < n) {
                        const float *v = reinterpret_cast<const float *>(shq) + 3 * lane;
                        float yv[16];
                        real_sh_upto<LSH>(v[0], v[1], v[2], prm.vec_mode == 1, yv);
#pragma unroll
                        for (int j = 0; j < SHN; ++j) Y[lane * SHN + j] = yv[j];
                    }
                    __syncwarp();
                    shq = reinterpret_cast<const unsigned char *>(Y);
                }
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
                            if constexpr (LV::kEdgePair) mo[64 * k + (q & 1)] = v;
                            else if constexpr (LV::kPair) *reinterpret_cast<float2 *>(mo + 64 * k) = make_float2(v, v);
                            else mo[32 * k] = v;
                        }
                    }
                    shq += SHN * 4;
                    if (!LV::kEdgePair || (q & 1)) mo += MS;  // edge pairs: one block per two edges
                }
            }
            __syncwarp();
            const FT *wl = reinterpret_cast<const FT *>(sb) + ch0;
            const FT *xl = reinterpret_cast<const FT *>(sb + prm.f_off) + ch0;
            if constexpr (kMlpReg) {
                // this lane's weights of every edge of the chunk and path, paired
                // by edge: wp[j][t] = (w[2j][t], w[2j+1][t]) with
                // w[q][t] = b2[t][c] + sum_i w2[i][t][c] h[i][q], the sum in order of i
                const ulonglong2 *h2 = reinterpret_cast<const ulonglong2 *>(base + prm.h_off);
                // (w2[i][t][c], w2[i][t][c]) for t < P.n (i = kMlpHidden: the bias)
                auto w2_pairs = [&](int i, f32x2 (&ww)[8]) {
                    if constexpr (kMlpSplat) {
                        const ulonglong2 *w2v = reinterpret_cast<const ulonglong2 *>(smem + prm.w2s_off) + lane;
#pragma unroll
                        for (int jj = 0; jj < (P.n + 1) / 2; ++jj) {
                            const ulonglong2 u = w2v[(i * 4 + jj) * 32];
                            ww[2 * jj] = u.x;
                            ww[2 * jj + 1] = u.y;
                        }
                    } else {
                        const float4 *w2v = reinterpret_cast<const float4 *>(smem + prm.w2s_off) + lane;
#pragma unroll
                        for (int hh = 0; hh < (P.n + 3) / 4; ++hh) {
                            const float4 u = w2v[(i * 2 + hh) * 32];
                            ww[4 * hh] = pack2(u.x, u.x);
                            ww[4 * hh + 1] = pack2(u.y, u.y);
                            ww[4 * hh + 2] = pack2(u.z, u.z);
                            ww[4 * hh + 3] = pack2(u.w, u.w);
                        }
                    }
                };
                f32x2 wp[kMlpChunk / 2][P.n];
                {
                    f32x2 bb[8];
                    w2_pairs(kMlpHidden, bb);
#pragma unroll
                    for (int j = 0; j < kMlpChunk / 2; ++j)
#pragma unroll
                        for (int t = 0; t < P.n; ++t) wp[j][t] = bb[t];
                }
#pragma unroll
                for (int i = 0; i < kMlpHidden; ++i) {
                    f32x2 ww[8];
                    w2_pairs(i, ww);
                    const ulonglong2 ha = h2[2 * i], hb = h2[2 * i + 1];
                    const f32x2 hp[4] = {ha.x, ha.y, hb.x, hb.y};
#pragma unroll
                    for (int j = 0; j < kMlpChunk / 2; ++j)
#pragma unroll
                        for (int t = 0; t < P.n; ++t) vfma(wp[j][t], ww[t], hp[j]);
                }
                // edges (q, q+1) of an aligned pair together when they share the
                // destination, else one at a time with the other half zeroed
                static_for<kMlpChunk / 2>([&](auto jc) {
                    constexpr int j = decltype(jc)::value, q = 2 * j;
                    if (q < n) {
                        const float *Mq = Mw + j * MS;
                        const FT *xa = xl + q * DX;
                        const bool has_b = q + 1 < n;
                        const FT *xb = has_b ? xa + DX : xa;
                        bool pa = true, pb = has_b;  // edges of the pair still to add
                        while (pa || pb) {
                            while (e >= seg_end && cur_d < d_end) {
                                store_row(cur_d);
                                ++cur_d;
                                enter(cur_d);
                            }
                            const bool ua = pa, ub = pb && (!pa || e + 1 < seg_end);
                            V xr[RI][1], wv[P.n][1];
#pragma unroll
                            for (int r = 0; r < RI; ++r) xr[r][0] = pack2(to_float(xa[r * MUL]), to_float(xb[r * MUL]));
#pragma unroll
                            for (int t = 0; t < P.n; ++t) wv[t][0] = wp[j][t];
                            if (!(ua && ub)) {  // one edge of the pair: the other half adds zero
#pragma unroll
                                for (int r = 0; r < RI; ++r)
                                    xr[r][0] = pack2(ua ? lo_f(xr[r][0]) : 0.f, ub ? hi_f(xr[r][0]) : 0.f);
#pragma unroll
                                for (int t = 0; t < P.n; ++t)
                                    wv[t][0] = pack2(ua ? lo_f(wv[t][0]) : 0.f, ub ? hi_f(wv[t][0]) : 0.f);
                            }
                            static_for<P.n>([&](auto tc) {
                                constexpr int T = decltype(tc)::value;
                                ring_path_w<LI, LSH, LO, T, CPT, PK>(acc, xr, wv[T], Mq);
                            });
                            e += (int)ua + (int)ub;
                            pa = false;
                            pb = pb && !ub;
                        }
                    }
                });
            } else if constexpr (LV::kEdgePair) {
                // edges (q, q+1) of an aligned pair together when they share the
                // destination, else one at a time with the other half zeroed
                for (int q = 0; q < n; q += 2) {
                    while (e >= seg_end && cur_d < d_end) {
                        store_row(cur_d);
                        ++cur_d;
                        enter(cur_d);
                    }
                    const float *Mq = Mw + (q >> 1) * MS;
                    const FT *xa = xl + q * (FB / (int)sizeof(FT)), *wa = wl + q * (WB / (int)sizeof(FT));
                    // the second slot only when it holds an edge of this chunk
                    const bool has_b = q + 1 < n;
                    const FT *xb = has_b ? xa + FB / (int)sizeof(FT) : xa;
                    const FT *wb2 = has_b ? wa + WB / (int)sizeof(FT) : wa;
                    auto run = [&](bool use_a, bool use_b) {
                        V xr[RI][1];
#pragma unroll
                        for (int r = 0; r < RI; ++r) {
                            const float a = to_float(xa[r * MUL]), b = to_float(xb[r * MUL]);
                            xr[r][0] = pack2(use_a ? a : 0.f, use_b ? b : 0.f);
                        }
                        static_for<P.n>([&](auto tc) {
                            ring_path<LI, LSH, LO, decltype(tc)::value, CPT, PK, FT>(acc, xr, wa, wb2, Mq, use_a, use_b);
                        });
                    };
                    if (has_b && e + 1 < seg_end) {
                        run(true, true);
                        e += 2;
                    } else {
                        run(true, false);
                        ++e;
                        if (has_b) {
                            while (e >= seg_end && cur_d < d_end) {
                                store_row(cur_d);
                                ++cur_d;
                                enter(cur_d);
                            }
                            run(false, true);
                            ++e;
                        }
                    }
                }
            } else {
                for (int q = 0; q < n; ++q, ++e) {
                    while (e >= seg_end && cur_d < d_end) {
                        store_row(cur_d);
                        ++cur_d;
                        enter(cur_d);
                    }
                    const FT *xq = xl + q * (FB / (int)sizeof(FT));
                    V xr[RI][NV];
#pragma unroll
                    for (int r = 0; r < RI; ++r) load_lane<CPT, PK>(xq + r * MUL, xr[r]);
                    const float *Mq = Mw + q * MS;
                    if constexpr (kMlpCols) {
                        // w[p][c] = b2[p][c] + sum_i w2[i][p][c] h[i], the sum in order of i
                        float hv[kMlpHidden];
                        const float4 *h4 = reinterpret_cast<const float4 *>(base + prm.h_off) + q * (kMlpHidden / 4);
#pragma unroll
                        for (int i4 = 0; i4 < kMlpHidden / 4; ++i4) {
                            const float4 t = h4[i4];
                            hv[4 * i4] = t.x;
                            hv[4 * i4 + 1] = t.y;
                            hv[4 * i4 + 2] = t.z;
                            hv[4 * i4 + 3] = t.w;
                        }
                        static_for<P.n>([&](auto tc) {
                            constexpr int T = decltype(tc)::value;
                            float ws[CPT];
                            ldg_lane<CPT>(prm.mlp_b2 + T * MUL + ch0, ws);
#pragma unroll
                            for (int i = 0; i < kMlpHidden; ++i) {
                                float w[CPT];
                                ldg_lane<CPT>(prm.mlp_w2 + i * WNUM + T * MUL + ch0, w);
#pragma unroll
                                for (int c = 0; c < CPT; ++c) ws[c] = fmaf(w[c], hv[i], ws[c]);
                            }
                            V wv[NV];
#pragma unroll
                            for (int c = 0; c < NV; ++c) {
                                if constexpr (LV::kPair) wv[c] = pack2(ws[2 * c], ws[2 * c + 1]);
                                else wv[c] = ws[c];
                            }
                            ring_path_w<LI, LSH, LO, T, CPT, PK>(acc, xr, wv, Mq);
                        });
                    } else {
                        const FT *wq = wl + q * (WB / (int)sizeof(FT));
                        static_for<P.n>([&](auto tc) {
                            ring_path<LI, LSH, LO, decltype(tc)::value, CPT, PK, FT>(acc, xr, wq, wq, Mq);
                        });
                    }
                }
            }
            // this warp's reads of the stage come before the bulk copies that refill it
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
        if (lane == 0) {
            set_status(prm.status, TP_DEV_ERR_TIMEOUT);
            // the partial rows of the piece that failed and of the pieces never
            // reached are not written: the merge must skip them
            for (int j2 = failed_j; j2 < np_w; ++j2) {
                prm.carry_dst[2 * (gw + j2 * nW)] = -1;
                prm.carry_dst[2 * (gw + j2 * nW) + 1] = -1;
            }
        }
        // let the copies still in flight land (full time limit) before the
        // shared memory is released
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
