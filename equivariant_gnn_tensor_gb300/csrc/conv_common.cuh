// Shared pieces of the warp-per-segment convolution kernels (forward and the
// source-side backward): per-warp shared-memory pipeline layout, the chunk
// iterator over a warp's segments, the per-edge M build and the per-path
// register contractions.
#pragma once
#include "common.cuh"

namespace tpc {

// (l+1)^2 rows: the slot of degree l occupies rows [l*l, (l+1)*(l+1)).
__host__ __device__ constexpr int rows_upto(int l) { return (l + 1) * (l + 1); }

struct ChunkMeta {
    int32_t seg;    // segment (destination row for the forward)
    int32_t e0;     // first edge slot of the chunk
    int32_t n;      // edges in the chunk (0 for an empty segment)
    uint32_t bits;  // bit0 valid, bit1 first of segment, bit2 last of segment; bits 8.. edge-valid mask
};
constexpr uint32_t kValid = 1u, kFirst = 2u, kLast = 4u;

// Per-warp shared memory: S mbarriers, S chunk records, S stage buffers, one M buffer.
struct WarpLayout {
    int stages;
    int eps;          // edges per chunk
    int w_bytes;      // one edge's weight row
    int f_bytes;      // one gathered feature row
    int sh_floats;    // one edge's harmonic row
    int stage_bytes;  // eps*(w_bytes + f_bytes) + sh (rounded to 128)
    int w_off, f_off, sh_off;  // inside a stage
    int m_floats;     // eps*R
    int q_floats;     // edge-gradient mode: R*33 partials + R reduced values (else 0)
    int head_bytes;   // barriers + chunk records (rounded to 128)
    int warp_bytes;   // total per warp (multiple of 128)
};

inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

inline WarpLayout make_layout(int stages, int eps, int w_bytes, int f_bytes, int sh_floats, int R,
                              bool edge_grad = false) {
    WarpLayout L;
    L.stages = stages;
    L.eps = eps;
    L.w_bytes = w_bytes;
    L.f_bytes = f_bytes;
    L.sh_floats = sh_floats;
    L.w_off = 0;
    L.f_off = eps * w_bytes;
    L.sh_off = L.f_off + eps * f_bytes;
    L.stage_bytes = round_up(L.sh_off + eps * sh_floats * 4, 128);
    L.m_floats = eps * R;
    L.q_floats = edge_grad ? R * 34 : 0;
    L.head_bytes = round_up(stages * (8 + (int)sizeof(ChunkMeta)), 128);
    L.warp_bytes = round_up(L.head_bytes + stages * L.stage_bytes + (L.m_floats + L.q_floats) * 4, 128);
    return L;
}

constexpr int kTablesBytes = (int)((sizeof(SmemTables) + 127) / 128 * 128);

// Transposed recipe (harmonic gradient), edge-gradient mode only.
struct SmemTrTables {
    uint16_t tr_ptr[kMaxSh + 1];
    uint16_t tr_r[kMaxTerms];
    float tr_c[kMaxTerms];
};
constexpr int kTrTablesBytes = (int)((sizeof(SmemTrTables) + 127) / 128 * 128);

// Build M for the n edges of a chunk: M[q*R + r] = sum_t coef_t * sh[q][j_t].
__device__ __forceinline__ void build_m(const SmemTables *st, const float *sh_stage, int sh_floats, int n,
                                        int R, float *M, int lane) {
    for (int q = 0; q < n; ++q) {
        const float *shq = sh_stage + q * sh_floats;
        for (int r = lane; r < R; r += 32) {
            float acc = 0.f;
            const int t1 = st->rec_ptr[r + 1];
            for (int t = st->rec_ptr[r]; t < t1; ++t) acc = fmaf(st->rec_c[t], shq[st->rec_j[t]], acc);
            M[q * R + r] = acc;
        }
    }
}

// Load the (2LA+1)*(2LC+1) floats of one path's M block (16-byte aligned).
template <int NM>
__device__ __forceinline__ void load_m(const float *Mp, float (&m)[(NM + 3) / 4 * 4]) {
    const float4 *M4 = reinterpret_cast<const float4 *>(Mp);
#pragma unroll
    for (int q = 0; q < (NM + 3) / 4; ++q) {
        float4 t = M4[q];
        m[4 * q + 0] = t.x;
        m[4 * q + 1] = t.y;
        m[4 * q + 2] = t.z;
        m[4 * q + 3] = t.w;
    }
}

// Forward contraction of one path for CPT channels:
//   acc[lc^2 + k][c] += w[c] * sum_i M[i][k] * x[la^2 + i][c]
template <int LA, int LC, int RI, int RO, int CPT>
__device__ __forceinline__ void path_fwd(float (&acc)[RO][CPT], const float (&xr)[RI][CPT], const float (&wv)[CPT],
                                         const float *Mp) {
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NM = NA * NC;
    float m[(NM + 3) / 4 * 4];
    load_m<NM>(Mp, m);
    if constexpr (NA <= NC) {
        float wx[NA][CPT];
#pragma unroll
        for (int i = 0; i < NA; ++i)
#pragma unroll
            for (int c = 0; c < CPT; ++c) wx[i][c] = wv[c] * xr[LA * LA + i][c];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float t = acc[LC * LC + k][c];
#pragma unroll
                for (int i = 0; i < NA; ++i) t = fmaf(m[i * NC + k], wx[i][c], t);
                acc[LC * LC + k][c] = t;
            }
    } else {
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float t = m[k] * xr[LA * LA][c];
#pragma unroll
                for (int i = 1; i < NA; ++i) t = fmaf(m[i * NC + k], xr[LA * LA + i][c], t);
                acc[LC * LC + k][c] = fmaf(wv[c], t, acc[LC * LC + k][c]);
            }
    }
}

// Source-side backward contraction of one path for CPT channels:
//   acc[la^2 + i][c] += w[c] * sum_k M[i][k] * g[lc^2 + k][c]
template <int LA, int LC, int RI, int RO, int CPT>
__device__ __forceinline__ void path_bwd_x(float (&acc)[RI][CPT], const float (&gr)[RO][CPT], const float (&wv)[CPT],
                                           const float *Mp) {
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NM = NA * NC;
    float m[(NM + 3) / 4 * 4];
    load_m<NM>(Mp, m);
    if constexpr (NC <= NA) {
        float wg[NC][CPT];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int c = 0; c < CPT; ++c) wg[k][c] = wv[c] * gr[LC * LC + k][c];
#pragma unroll
        for (int i = 0; i < NA; ++i)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float t = acc[LA * LA + i][c];
#pragma unroll
                for (int k = 0; k < NC; ++k) t = fmaf(m[i * NC + k], wg[k][c], t);
                acc[LA * LA + i][c] = t;
            }
    } else {
#pragma unroll
        for (int i = 0; i < NA; ++i)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float t = m[i * NC] * gr[LC * LC][c];
#pragma unroll
                for (int k = 1; k < NC; ++k) t = fmaf(m[i * NC + k], gr[LC * LC + k][c], t);
                acc[LA * LA + i][c] = fmaf(wv[c], t, acc[LA * LA + i][c]);
            }
    }
}

// Edge gradients of one path for CPT channels:
//   dw[c]      = sum_i x[la^2+i][c] * sum_k M[i][k] g[lc^2+k][c]
//   Q[i][k]   += sum_c w[c] x[la^2+i][c] g[lc^2+k][c]   (this lane's channels; reduced across lanes later)
// Qcol points at this lane's column of the path's partial block (row stride 33).
template <int LA, int LC, int RI, int RO, int CPT>
__device__ __forceinline__ void path_bwd_edge(const float (&xr)[RI][CPT], const float (&gr)[RO][CPT],
                                              const float (&wv)[CPT], const float *Mp, float (&dwv)[CPT],
                                              float *Qcol) {
    constexpr int NA = 2 * LA + 1, NC = 2 * LC + 1, NM = NA * NC;
    float m[(NM + 3) / 4 * 4];
    load_m<NM>(Mp, m);
#pragma unroll
    for (int c = 0; c < CPT; ++c) dwv[c] = 0.f;
#pragma unroll
    for (int i = 0; i < NA; ++i)
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            float t = m[i * NC] * gr[LC * LC][c];
#pragma unroll
            for (int k = 1; k < NC; ++k) t = fmaf(m[i * NC + k], gr[LC * LC + k][c], t);
            dwv[c] = fmaf(xr[LA * LA + i][c], t, dwv[c]);
        }
#pragma unroll
    for (int i = 0; i < NA; ++i) {
        float wx[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) wx[c] = wv[c] * xr[LA * LA + i][c];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            float q = wx[0] * gr[LC * LC + k][0];
#pragma unroll
            for (int c = 1; c < CPT; ++c) q = fmaf(wx[c], gr[LC * LC + k][c], q);
            Qcol[(i * NC + k) * 33] = q;
        }
    }
}

}  // namespace tpc
