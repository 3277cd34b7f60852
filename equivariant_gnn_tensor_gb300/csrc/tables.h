// Internal descriptor layout shared by the host builder and the kernels.
//
// The per-edge work is split in two. What depends only on the edge's
// harmonics is folded once per edge into small matrices
//     M_p[i][k] = sum_j C_p[i,j,k] * sh[e, b_p, j]        (one per path p)
// and what depends on the channel u is then a dense (2la+1)x(2lc+1)
// mat-vec per path and channel:
//     out[c_p, k, u] += w[e,p,u] * sum_i M_p[i][k] * x[src, a_p, i, u].
// M is laid out path after path, each path's block (i-major, k-minor)
// padded to a multiple of 4 floats so it can be read with 16-byte loads.
// The "recipe" lists, for every M entry r, the (harmonic index, coefficient)
// terms of its sum; the transposed recipe gives the harmonic gradient
//     dsh[j] = sum_r G[r][j] * Q[r],  Q_p[i][k] = sum_u w_p x_i g_k.
#pragma once
#include <cstdint>

namespace tpc {

constexpr int kMaxPaths = 64;
constexpr int kMaxM = 768;      // M floats per edge over all paths (padded)
constexpr int kMaxTerms = 640;  // nonzero Clebsch-Gordan entries over all paths
constexpr int kMaxSh = 64;      // harmonic row width
constexpr int kMaxShBlocks = 16;
constexpr int kMaxL = 3;

struct Tables {
    int32_t n_paths, mul, dim_x, dim_sh, dim_out, wnum;
    int32_t R;    // M floats per edge
    int32_t nnz;  // recipe terms
    int32_t x_off[4];  // offset of the input block of degree l (-1: none)
    int32_t o_off[4];  // offset of the output block of degree l (-1: none)
    int32_t n_sh_blocks;
    uint8_t sh_l[kMaxShBlocks];
    uint8_t la[kMaxPaths], lb[kMaxPaths], lc[kMaxPaths], pad0[kMaxPaths];
    uint16_t m_off[kMaxPaths];
    uint16_t rec_ptr[kMaxM + 1];
    uint16_t rec_j[kMaxTerms];
    float rec_c[kMaxTerms];
    uint16_t tr_ptr[kMaxSh + 1];
    uint16_t tr_r[kMaxTerms];
    float tr_c[kMaxTerms];
};

// Runtime tables for a compile-time path program (program.h): valid when the
// descriptor's paths are exactly the program's and every nonzero
// Clebsch-Gordan entry lies inside the program's M pattern.
struct ProgramPlan {
    int32_t valid;
    int32_t shape;   // index into kProgShapes
    int32_t R, nnz;
    int16_t wofs[32];  // weight-row offset (elements) of program path t
    // M entry r (program layout) = ec[r][0] * sh[ej[r] & 0xffff] + ec[r][1] * sh[ej[r] >> 16]
    uint32_t ej[kMaxM];
    float ec[kMaxM][2];
};

}  // namespace tpc

namespace tpc {
// Drop the launch plans cached for descriptor `uid` (called when it is destroyed).
void launch_cache_forget(uint64_t uid);
}  // namespace tpc

struct tp_desc {
    uint64_t uid;  // unique per descriptor created in this process (launch-plan cache key)
    int layout;    // tp_layout of the feature rows the caller passes (the kernels compute in ir_mul)
    int unsimp;    // one output block per path (tp_desc_create_unsimplified)
    int unsimp_dim_out;                 // sum over paths of mul*(2lc+1)
    int unsimp_off[tpc::kMaxPaths];     // offset of path p's output block
    int unsimp_block[tpc::kMaxPaths];   // position of path p's block in the output listing
    // parsed irreps: (mul, l, parity) with parity +1/-1 (O3) or 0 (SO3)
    int n_in, n_sh, n_out;
    int in_mul[8], in_l[8], in_p[8];
    int sh_l[tpc::kMaxShBlocks], sh_p[tpc::kMaxShBlocks];
    int out_mul[8], out_l[8], out_p[8];
    int in_off[8], sh_off[tpc::kMaxShBlocks], out_off[8];
    int lmax_in, lmax_sh, lmax_out;
    int n_paths;
    int path_a[tpc::kMaxPaths], path_b[tpc::kMaxPaths], path_c[tpc::kMaxPaths];
    double *cg[tpc::kMaxPaths];  // dense [2la+1][2lb+1][2lc+1]
    tpc::Tables tab;
    tpc::ProgramPlan prog;
};
