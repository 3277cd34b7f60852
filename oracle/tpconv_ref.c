/* fp64 CPU oracle of the channelwise (uvu) tensor-product convolution, plain C
 * loops with OpenMP over destination rows (forward), edges (dw, dsh) and source
 * rows (dx). TEST INFRASTRUCTURE ONLY: the library never links or calls this.
 *
 * It restates, loop for loop, the sums of the channelwise tensor product with
 * gather and sum-scatter (Lesson 12a: Foundations of cuEquivariance, section
 * 21.4, "[ijk]·a[uv]·b[iu]·c[jv] -> D[kuv]" with v = 1; "cuEquivariance in
 * PyTorch", SegmentedPolynomial: gather and scatter):
 *
 *   out[d,c,k,u] = sum_{e in seg(d)} sum_p w[e,p,u] sum_{i,j} C_p[i,j,k] x[src[e],a,i,u] sh[e,b,j]
 *
 * and its exact backward. Feature rows are in the ir_mul layout: element (i,u)
 * of a block at offset off is off + i*mul + u. The Clebsch-Gordan tensors come
 * in from the Python oracle (oracle/so3.py), dense [2la+1][2lb+1][2lc+1] per
 * path; entries that are exactly zero are skipped (they add exactly zero).
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* path_info: per path 6 ints: la, lb, lc, off_a, off_b, off_c.
 * cg_off: start of path p's dense tensor in cg. */

static void edge_message_add(int n_paths, const int32_t *pi, const double *cg, const int64_t *cg_off,
                             int mul, const double *xs, const double *she, const double *we,
                             double *acc)
{
    for (int p = 0; p < n_paths; ++p) {
        const int la = pi[6 * p + 0], lb = pi[6 * p + 1], lc = pi[6 * p + 2];
        const int oa = pi[6 * p + 3], ob = pi[6 * p + 4], oc = pi[6 * p + 5];
        const int na = 2 * la + 1, nb = 2 * lb + 1, nc = 2 * lc + 1;
        const double *C = cg + cg_off[p];
        const double *wp = we + (int64_t)p * mul;
        for (int i = 0; i < na; ++i)
            for (int j = 0; j < nb; ++j)
                for (int k = 0; k < nc; ++k) {
                    const double cijk = C[(i * nb + j) * nc + k];
                    if (cijk == 0.0) continue;
                    const double cs = cijk * she[ob + j];
                    const double *xi = xs + oa + (int64_t)i * mul;
                    double *ok = acc + oc + (int64_t)k * mul;
                    for (int u = 0; u < mul; ++u) ok[u] += wp[u] * cs * xi[u];
                }
    }
}

/* Forward for the destination rows listed in `rows` (all rows when rows == NULL,
 * n_list = n_dst). Edges are in dst-sorted order described by row_ptr. */
void ref_conv_forward(int n_paths, const int32_t *path_info, const double *cg, const int64_t *cg_off,
                      int mul, int dim_x, int dim_sh, int dim_out, int weight_numel,
                      const double *x, const double *sh, const double *w, const int32_t *src,
                      const int64_t *row_ptr, int n_dst, const int32_t *rows, int n_list,
                      double *out, int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#endif
    (void)n_dst;
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n_list; ++r) {
        const int d = rows ? rows[r] : r;
        double *o = out + (int64_t)r * dim_out;
        memset(o, 0, sizeof(double) * (size_t)dim_out);
        for (int64_t e = row_ptr[d]; e < row_ptr[d + 1]; ++e)
            edge_message_add(n_paths, path_info, cg, cg_off, mul, x + (int64_t)src[e] * dim_x,
                             sh + e * dim_sh, w + e * weight_numel, o);
    }
}

/* dw and dsh for the edges listed in `edges` (all when NULL). */
void ref_conv_backward_edges(int n_paths, const int32_t *pi, const double *cg, const int64_t *cg_off,
                             int mul, int dim_x, int dim_sh, int dim_out, int weight_numel,
                             const double *x, const double *sh, const double *w, const double *g,
                             const int32_t *src, const int32_t *dst, const int64_t *edges, int64_t n_list,
                             double *dw, double *dsh, int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#endif
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < n_list; ++r) {
        const int64_t e = edges ? edges[r] : r;
        const double *xs = x + (int64_t)src[e] * dim_x;
        const double *gd = g + (int64_t)dst[e] * dim_out;
        const double *she = sh + e * dim_sh;
        const double *we = w + e * weight_numel;
        double *dwe = dw + r * weight_numel;
        double *dshe = dsh + r * dim_sh;
        memset(dwe, 0, sizeof(double) * (size_t)weight_numel);
        memset(dshe, 0, sizeof(double) * (size_t)dim_sh);
        for (int p = 0; p < n_paths; ++p) {
            const int la = pi[6 * p + 0], lb = pi[6 * p + 1], lc = pi[6 * p + 2];
            const int oa = pi[6 * p + 3], ob = pi[6 * p + 4], oc = pi[6 * p + 5];
            const int na = 2 * la + 1, nb = 2 * lb + 1, nc = 2 * lc + 1;
            const double *C = cg + cg_off[p];
            for (int i = 0; i < na; ++i)
                for (int j = 0; j < nb; ++j)
                    for (int k = 0; k < nc; ++k) {
                        const double cijk = C[(i * nb + j) * nc + k];
                        if (cijk == 0.0) continue;
                        const double *xi = xs + oa + (int64_t)i * mul;
                        const double *gk = gd + oc + (int64_t)k * mul;
                        const double *wp = we + (int64_t)p * mul;
                        double *dwp = dwe + (int64_t)p * mul;
                        double sj = 0.0;
                        for (int u = 0; u < mul; ++u) {
                            dwp[u] += cijk * xi[u] * she[ob + j] * gk[u];
                            sj += cijk * xi[u] * wp[u] * gk[u];
                        }
                        dshe[ob + j] += sj;
                    }
        }
    }
}

/* dx for the source rows listed in `rows` (all when NULL); the edges of source
 * s are src_perm[src_row_ptr[s] .. src_row_ptr[s+1]). */
void ref_conv_backward_dx(int n_paths, const int32_t *pi, const double *cg, const int64_t *cg_off,
                          int mul, int dim_x, int dim_sh, int dim_out, int weight_numel,
                          const double *sh, const double *w, const double *g, const int32_t *dst,
                          const int32_t *src_perm, const int64_t *src_row_ptr, const int32_t *rows,
                          int n_list, double *dx, int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#endif
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n_list; ++r) {
        const int s = rows ? rows[r] : r;
        double *dxs = dx + (int64_t)r * dim_x;
        memset(dxs, 0, sizeof(double) * (size_t)dim_x);
        for (int64_t t = src_row_ptr[s]; t < src_row_ptr[s + 1]; ++t) {
            const int64_t e = src_perm[t];
            const double *gd = g + (int64_t)dst[e] * dim_out;
            const double *she = sh + e * dim_sh;
            const double *we = w + e * weight_numel;
            for (int p = 0; p < n_paths; ++p) {
                const int la = pi[6 * p + 0], lb = pi[6 * p + 1], lc = pi[6 * p + 2];
                const int oa = pi[6 * p + 3], ob = pi[6 * p + 4], oc = pi[6 * p + 5];
                const int na = 2 * la + 1, nb = 2 * lb + 1, nc = 2 * lc + 1;
                const double *C = cg + cg_off[p];
                const double *wp = we + (int64_t)p * mul;
                for (int i = 0; i < na; ++i)
                    for (int j = 0; j < nb; ++j)
                        for (int k = 0; k < nc; ++k) {
                            const double cijk = C[(i * nb + j) * nc + k];
                            if (cijk == 0.0) continue;
                            const double cs = cijk * she[ob + j];
                            const double *gk = gd + oc + (int64_t)k * mul;
                            double *di = dxs + oa + (int64_t)i * mul;
                            for (int u = 0; u < mul; ++u) di[u] += wp[u] * cs * gk[u];
                        }
            }
        }
    }
}

int ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
