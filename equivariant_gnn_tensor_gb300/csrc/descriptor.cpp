// Host-side descriptor builder: irreps strings -> path table, real
// Clebsch-Gordan tensors and the kernel tables (tables.h).
//
// Irreps grammar and dims: Lesson 12a: Foundations of cuEquivariance,
// section 21.2. Path rule and weight order: section 21.4 (channelwise
// "uvu" paths filtered by the requested output types). The real
// Clebsch-Gordan tensors are derived here from Racah's closed formula for
// the complex coefficients <l1 m1 l2 m2 | l3 m3>, mapped to the real basis
// (m = -l..l, z pole, cos-type for m > 0, sin-type for m < 0) by the unitary
// U_l with Y_real = U_l Y_complex:
//     C[i,j,k] = sum U3[k,M] <l1 m1 l2 m2|l3 M> conj(U1[i,m1]) conj(U2[j,m2]),
// which is real up to one global phase; the phase is dropped, the tensor is
// scaled to be orthonormal over (i,j) for each k and its sign fixed so the
// first entry above 1e-9 in (i,j,k) row-major order is positive.
#include <algorithm>
#include <atomic>
#include <cctype>
#include <cmath>
#include <complex>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/tpconv.h"
#include "program.h"
#include "symc.h"
#include "tables.h"

namespace {

struct Term {
    int mul, l, p;
};

// Parse "32x0e + 32x1o" / "0+1+2". Returns false on a malformed string.
bool parse_irreps(const char *s, std::vector<Term> &out) {
    out.clear();
    std::string body;
    for (const char *c = s; *c; ++c)
        if (!std::isspace(static_cast<unsigned char>(*c))) body.push_back(*c);
    if (body.empty()) return false;
    int with_parity = 0, without = 0;
    size_t pos = 0;
    while (pos <= body.size()) {
        size_t plus = body.find('+', pos);
        std::string t = body.substr(pos, plus == std::string::npos ? std::string::npos : plus - pos);
        if (t.empty()) return false;
        Term term{1, 0, 0};
        size_t x = t.find('x');
        std::string lp = t;
        if (x != std::string::npos) {
            std::string m = t.substr(0, x);
            if (m.empty() || m.size() > 6) return false;
            for (char ch : m)
                if (!std::isdigit(static_cast<unsigned char>(ch))) return false;
            term.mul = std::atoi(m.c_str());
            lp = t.substr(x + 1);
        }
        if (lp.empty()) return false;
        char last = lp.back();
        if (last == 'e' || last == 'o') {
            term.p = last == 'e' ? 1 : -1;
            lp.pop_back();
            ++with_parity;
        } else {
            ++without;
        }
        if (lp.empty() || lp.size() > 3) return false;
        for (char ch : lp)
            if (!std::isdigit(static_cast<unsigned char>(ch))) return false;
        term.l = std::atoi(lp.c_str());
        out.push_back(term);
        if (plus == std::string::npos) break;
        pos = plus + 1;
    }
    return !(with_parity && without);
}

double fact(int n) {
    double r = 1.0;
    for (int i = 2; i <= n; ++i) r *= i;
    return r;
}

// <j1 m1 j2 m2 | J M>, Racah's formula.
double cg_complex(int j1, int m1, int j2, int m2, int J, int M) {
    if (M != m1 + m2 || J < std::abs(j1 - j2) || J > j1 + j2) return 0.0;
    if (std::abs(m1) > j1 || std::abs(m2) > j2 || std::abs(M) > J) return 0.0;
    double pre = std::sqrt((2.0 * J + 1.0) * fact(J + j1 - j2) * fact(J - j1 + j2) * fact(j1 + j2 - J) /
                           fact(j1 + j2 + J + 1));
    pre *= std::sqrt(fact(J + M) * fact(J - M) * fact(j1 - m1) * fact(j1 + m1) * fact(j2 - m2) * fact(j2 + m2));
    double s = 0.0;
    for (int k = 0; k <= j1 + j2 + J + 1; ++k) {
        int a[6] = {k, j1 + j2 - J - k, j1 - m1 - k, j2 + m2 - k, J - j2 + m1 + k, J - j1 - m2 + k};
        bool ok = true;
        for (int v : a) ok = ok && v >= 0;
        if (!ok) continue;
        double den = 1.0;
        for (int v : a) den *= fact(v);
        s += ((k & 1) ? -1.0 : 1.0) / den;
    }
    return pre * s;
}

// U_l[row = m+l][col = m'+l]: real harmonic m as a combination of complex m'.
std::vector<std::complex<double>> real_basis(int l) {
    const int n = 2 * l + 1;
    std::vector<std::complex<double>> u(n * n, 0.0);
    const double r2 = 1.0 / std::sqrt(2.0);
    for (int m = -l; m <= l; ++m) {
        const int row = m + l;
        if (m > 0) {
            u[row * n + (m + l)] = ((m & 1) ? -r2 : r2);
            u[row * n + (-m + l)] = r2;
        } else if (m < 0) {
            const int mu = -m;
            u[row * n + (-mu + l)] = std::complex<double>(0.0, r2);
            u[row * n + (mu + l)] = std::complex<double>(0.0, (mu & 1) ? r2 : -r2);
        } else {
            u[row * n + l] = 1.0;
        }
    }
    return u;
}

void real_cg(int l1, int l2, int l3, double *C) {
    const int n1 = 2 * l1 + 1, n2 = 2 * l2 + 1, n3 = 2 * l3 + 1;
    auto U1 = real_basis(l1), U2 = real_basis(l2), U3 = real_basis(l3);
    std::vector<std::complex<double>> T(n1 * n2 * n3, 0.0);
    for (int i = 0; i < n1; ++i)
        for (int j = 0; j < n2; ++j)
            for (int k = 0; k < n3; ++k) {
                std::complex<double> acc = 0.0;
                for (int m1 = -l1; m1 <= l1; ++m1) {
                    const auto a = std::conj(U1[i * n1 + (m1 + l1)]);
                    if (a == 0.0) continue;
                    for (int m2 = -l2; m2 <= l2; ++m2) {
                        const auto b = std::conj(U2[j * n2 + (m2 + l2)]);
                        if (b == 0.0) continue;
                        const int M = m1 + m2;
                        if (std::abs(M) > l3) continue;
                        const auto c = U3[k * n3 + (M + l3)];
                        if (c == 0.0) continue;
                        acc += c * a * b * cg_complex(l1, m1, l2, m2, l3, M);
                    }
                }
                T[(i * n2 + j) * n3 + k] = acc;
            }
    double nre = 0.0, nim = 0.0;
    for (auto &t : T) {
        nre += t.real() * t.real();
        nim += t.imag() * t.imag();
    }
    const bool use_re = nre >= nim;
    double norm2 = 0.0;
    for (size_t q = 0; q < T.size(); ++q) {
        C[q] = use_re ? T[q].real() : T[q].imag();
        norm2 += C[q] * C[q];
    }
    const double scale = norm2 > 0 ? std::sqrt(n3 / norm2) : 0.0;
    double sign = 0.0;
    for (size_t q = 0; q < T.size(); ++q) {
        C[q] *= scale;
        if (std::fabs(C[q]) < 1e-12) C[q] = 0.0;
        if (sign == 0.0 && std::fabs(C[q]) > 1e-9) sign = C[q] > 0 ? 1.0 : -1.0;
    }
    for (size_t q = 0; q < T.size(); ++q) C[q] *= sign;
}

// Match the descriptor against the compiled path programs (program.h) and
// build the program-layout recipe for the first one that fits.
void plan_program(tp_desc *d) {
    using namespace tpc;
    ProgramPlan &TP = d->prog;
    TP.valid = 0;
    for (int si = 0; si < kNumProgShapes; ++si) {
        const ProgShape sh = kProgShapes[si];
        const Program P = make_natural_program(sh.li, sh.lsh, sh.lo);
        if (P.n != d->n_paths || P.n > 32) continue;
        bool ok = true;
        for (int c = 0; c < d->n_out; ++c) ok = ok && d->out_l[c] <= sh.lo;
        for (int a = 0; a < d->n_in; ++a) ok = ok && d->in_l[a] <= sh.li;
        if (!ok) continue;
        int map[kProgMaxPaths];
        bool used[kMaxPaths] = {};
        for (int t = 0; t < P.n && ok; ++t) {
            map[t] = -1;
            for (int p = 0; p < d->n_paths; ++p) {
                if (used[p]) continue;
                if (d->in_l[d->path_a[p]] == P.p[t].la && d->sh_l[d->path_b[p]] == P.p[t].lb &&
                    d->out_l[d->path_c[p]] == P.p[t].lc) {
                    map[t] = p;
                    used[p] = true;
                    break;
                }
            }
            ok = map[t] >= 0;
        }
        if (!ok) continue;
        // every nonzero C[i,j,k] must have (i,k) inside the pattern
        for (int t = 0; t < P.n && ok; ++t) {
            const int p = map[t];
            const int la = P.p[t].la, lb = P.p[t].lb, lc = P.p[t].lc;
            const int n2 = 2 * lb + 1, n3 = 2 * lc + 1;
            for (int i = 0; i < 2 * la + 1 && ok; ++i)
                for (int k = 0; k < n3 && ok; ++k) {
                    bool nz = false;
                    for (int j = 0; j < n2; ++j) nz = nz || d->cg[p][(i * n2 + j) * n3 + k] != 0.0;
                    if (nz && !m_entry_possible(la, lb, lc, i, k)) ok = false;
                }
        }
        if (!ok || P.R > kMaxM) continue;
        int nnz = 0;
        for (int r = 0; r < P.R; ++r) {
            TP.ej[r] = 0;
            TP.ec[r][0] = TP.ec[r][1] = 0.f;
        }
        for (int t = 0; t < P.n && ok; ++t) {
            const int p = map[t];
            const int lb = P.p[t].lb, lc = P.p[t].lc;
            const int n2 = 2 * lb + 1, n3 = 2 * lc + 1;
            TP.wofs[t] = (int16_t)(p * d->tab.mul);
            for (int q = 0; q < P.nz[t]; ++q) {
                const int r = P.moff[t] + q;
                const int i = P.ik[t][q] >> 3, k = P.ik[t][q] & 7;
                int terms = 0;
                for (int j = 0; j < n2; ++j) {
                    const double c = d->cg[p][(i * n2 + j) * n3 + k];
                    if (c == 0.0) continue;
                    if (terms == 2) { ok = false; break; }
                    const uint32_t jg = (uint32_t)(d->sh_off[d->path_b[p]] + j);
                    TP.ej[r] |= terms == 0 ? jg : (jg << 16);
                    TP.ec[r][terms] = (float)c;
                    ++terms;
                    ++nnz;
                }
            }
        }
        if (!ok) continue;
        TP.R = P.R;
        TP.nnz = nnz;
        TP.shape = si;
        TP.valid = 1;
        return;
    }
}

void free_desc(tp_desc *d) {
    if (!d) return;
    tpc::launch_cache_forget(d->uid);
    for (int p = 0; p < d->n_paths; ++p) std::free(d->cg[p]);
    delete d;
}

}  // namespace

extern "C" tp_status tp_desc_create(const char *irreps_in, const char *irreps_sh, const char *irreps_out,
                                    tp_layout layout, tp_desc **out) {
    using namespace tpc;
    if (!irreps_in || !irreps_sh || !irreps_out || !out) return TP_ERR_ARG;
    *out = nullptr;
    std::vector<Term> tin, tsh, tout;
    if (!parse_irreps(irreps_in, tin) || !parse_irreps(irreps_sh, tsh) || !parse_irreps(irreps_out, tout))
        return TP_ERR_PARSE;
    if (layout != TP_IR_MUL && layout != TP_MUL_IR) return TP_ERR_ARG;
    // O3 vs SO3 must agree across the three strings
    auto kind = [](const std::vector<Term> &v) { return v[0].p != 0; };
    if (kind(tin) != kind(tsh) || kind(tin) != kind(tout)) return TP_ERR_PARSE;
    if (tin.size() > 4 || tout.size() > 4 || tsh.size() > (size_t)kMaxShBlocks) return TP_ERR_UNSUPPORTED;

    tp_desc *d = new (std::nothrow) tp_desc();
    if (!d) return TP_ERR_ARG;
    std::memset(d, 0, sizeof(*d));
    static std::atomic<uint64_t> next_uid{1};
    d->uid = next_uid.fetch_add(1);
    d->layout = (int)layout;
    d->n_in = (int)tin.size();
    d->n_sh = (int)tsh.size();
    d->n_out = (int)tout.size();
    int mul = tin[0].mul;
    bool seen_in[4] = {false, false, false, false}, seen_out[4] = {false, false, false, false};
    int off = 0;
    d->lmax_in = d->lmax_sh = d->lmax_out = 0;
    for (int a = 0; a < d->n_in; ++a) {
        const Term &t = tin[a];
        if (t.l > kMaxL || t.mul != mul || seen_in[t.l]) { free_desc(d); return TP_ERR_UNSUPPORTED; }
        seen_in[t.l] = true;
        d->in_mul[a] = t.mul; d->in_l[a] = t.l; d->in_p[a] = t.p; d->in_off[a] = off;
        off += t.mul * (2 * t.l + 1);
        if (t.l > d->lmax_in) d->lmax_in = t.l;
    }
    const int dim_x = off;
    off = 0;
    for (int b = 0; b < d->n_sh; ++b) {
        const Term &t = tsh[b];
        if (t.l > kMaxL || t.mul != 1) { free_desc(d); return TP_ERR_UNSUPPORTED; }
        d->sh_l[b] = t.l; d->sh_p[b] = t.p; d->sh_off[b] = off;
        off += 2 * t.l + 1;
        if (t.l > d->lmax_sh) d->lmax_sh = t.l;
    }
    const int dim_sh = off;
    off = 0;
    for (int c = 0; c < d->n_out; ++c) {
        const Term &t = tout[c];
        if (t.l > kMaxL || t.mul != mul || seen_out[t.l]) { free_desc(d); return TP_ERR_UNSUPPORTED; }
        seen_out[t.l] = true;
        d->out_mul[c] = t.mul; d->out_l[c] = t.l; d->out_p[c] = t.p; d->out_off[c] = off;
        off += t.mul * (2 * t.l + 1);
        if (t.l > d->lmax_out) d->lmax_out = t.l;
    }
    const int dim_out = off;
    if (mul % 8 != 0 || mul > 128 || mul <= 0 || dim_sh > kMaxSh) { free_desc(d); return TP_ERR_UNSUPPORTED; }

    // paths: a-major, then b, then l_o ascending (triangle rule, parity product)
    int np = 0;
    for (int a = 0; a < d->n_in; ++a)
        for (int b = 0; b < d->n_sh; ++b)
            for (int lo = std::abs(d->in_l[a] - d->sh_l[b]); lo <= d->in_l[a] + d->sh_l[b]; ++lo) {
                const int po = d->in_p[a] * d->sh_p[b];
                for (int c = 0; c < d->n_out; ++c) {
                    if (d->out_l[c] != lo || d->out_p[c] != po) continue;
                    if (np >= kMaxPaths) { free_desc(d); return TP_ERR_UNSUPPORTED; }
                    d->path_a[np] = a; d->path_b[np] = b; d->path_c[np] = c;
                    const int n1 = 2 * d->in_l[a] + 1, n2 = 2 * d->sh_l[b] + 1, n3 = 2 * lo + 1;
                    d->cg[np] = static_cast<double *>(std::malloc(sizeof(double) * n1 * n2 * n3));
                    if (!d->cg[np]) { free_desc(d); return TP_ERR_ARG; }
                    d->n_paths = np + 1;
                    real_cg(d->in_l[a], d->sh_l[b], lo, d->cg[np]);
                    ++np;
                }
            }
    d->n_paths = np;
    if (np == 0) { free_desc(d); return TP_ERR_UNSUPPORTED; }

    // kernel tables
    Tables &T = d->tab;
    T.n_paths = np; T.mul = mul; T.dim_x = dim_x; T.dim_sh = dim_sh; T.dim_out = dim_out;
    T.wnum = np * mul;
    for (int l = 0; l < 4; ++l) { T.x_off[l] = -1; T.o_off[l] = -1; }
    for (int a = 0; a < d->n_in; ++a) T.x_off[d->in_l[a]] = d->in_off[a];
    for (int c = 0; c < d->n_out; ++c) T.o_off[d->out_l[c]] = d->out_off[c];
    T.n_sh_blocks = d->n_sh;
    for (int b = 0; b < d->n_sh; ++b) T.sh_l[b] = (uint8_t)d->sh_l[b];
    int R = 0, nnz = 0;
    std::vector<std::vector<std::pair<int, float>>> col(dim_sh);  // transposed recipe
    for (int p = 0; p < np; ++p) {
        const int la = d->in_l[d->path_a[p]], lb = d->sh_l[d->path_b[p]], lc = d->out_l[d->path_c[p]];
        const int n1 = 2 * la + 1, n2 = 2 * lb + 1, n3 = 2 * lc + 1;
        T.la[p] = (uint8_t)la; T.lb[p] = (uint8_t)lb; T.lc[p] = (uint8_t)lc;
        T.m_off[p] = (uint16_t)R;
        const int padded = (n1 * n3 + 3) / 4 * 4;
        if (R + padded > kMaxM) { free_desc(d); return TP_ERR_UNSUPPORTED; }
        for (int q = 0; q < padded; ++q) {
            T.rec_ptr[R + q] = (uint16_t)nnz;
            if (q < n1 * n3) {
                const int i = q / n3, k = q % n3;
                for (int j = 0; j < n2; ++j) {
                    const double c = d->cg[p][(i * n2 + j) * n3 + k];
                    if (c == 0.0) continue;
                    if (nnz >= kMaxTerms) { free_desc(d); return TP_ERR_UNSUPPORTED; }
                    const int jg = d->sh_off[d->path_b[p]] + j;
                    T.rec_j[nnz] = (uint16_t)jg;
                    T.rec_c[nnz] = (float)c;
                    col[jg].push_back({R + q, (float)c});
                    ++nnz;
                }
            }
        }
        R += padded;
    }
    T.rec_ptr[R] = (uint16_t)nnz;
    T.R = R;
    T.nnz = nnz;
    int t = 0;
    for (int j = 0; j < dim_sh; ++j) {
        T.tr_ptr[j] = (uint16_t)t;
        for (auto &e : col[j]) { T.tr_r[t] = (uint16_t)e.first; T.tr_c[t] = e.second; ++t; }
    }
    T.tr_ptr[dim_sh] = (uint16_t)t;
    plan_program(d);
    *out = d;
    return TP_OK;
}

extern "C" tp_status tp_desc_create_unsimplified(const char *irreps_in, const char *irreps_sh,
                                                 const char *irreps_out, tp_layout layout, tp_desc **out) {
    if (layout != TP_IR_MUL) return TP_ERR_UNSUPPORTED;
    tp_status st = tp_desc_create(irreps_in, irreps_sh, irreps_out, layout, out);
    if (st != TP_OK) return st;
    tp_desc *d = *out;
    // blocks grouped by output type in the order of the output list, paths of one type in path order
    int off = 0, pos = 0;
    for (int c = 0; c < d->n_out; ++c)
        for (int p = 0; p < d->n_paths; ++p) {
            if (d->path_c[p] != c) continue;
            d->unsimp_off[p] = off;
            d->unsimp_block[p] = pos++;
            off += d->tab.mul * (2 * d->out_l[c] + 1);
        }
    d->unsimp_dim_out = off;
    d->unsimp = 1;
    return TP_OK;
}

extern "C" tp_status tp_desc_query(const tp_desc *d, tp_desc_info *info) {
    if (!d || !info) return TP_ERR_ARG;
    info->n_paths = d->n_paths;
    info->mul = d->tab.mul;
    info->dim_x = d->tab.dim_x;
    info->dim_sh = d->tab.dim_sh;
    info->dim_out = d->unsimp ? d->unsimp_dim_out : d->tab.dim_out;
    info->weight_numel = d->tab.wnum;
    info->n_in = d->n_in; info->n_sh = d->n_sh; info->n_out = d->unsimp ? d->n_paths : d->n_out;
    info->lmax_in = d->lmax_in; info->lmax_sh = d->lmax_sh; info->lmax_out = d->lmax_out;
    info->cg_nnz = d->tab.nnz;
    info->layout = d->layout;
    return TP_OK;
}

extern "C" tp_status tp_desc_path(const tp_desc *d, int32_t p, tp_path_info *info) {
    if (!d || !info || p < 0 || p >= d->n_paths) return TP_ERR_ARG;
    info->a = d->path_a[p]; info->b = d->path_b[p]; info->c = d->path_c[p];
    info->la = d->in_l[info->a]; info->lb = d->sh_l[info->b]; info->lc = d->out_l[info->c];
    if (d->unsimp) info->c = d->unsimp_block[p];
    return TP_OK;
}

extern "C" tp_status tp_desc_cg(const tp_desc *d, int32_t p, double *out, int64_t capacity) {
    if (!d || !out || p < 0 || p >= d->n_paths) return TP_ERR_ARG;
    const int la = d->in_l[d->path_a[p]], lb = d->sh_l[d->path_b[p]], lc = d->out_l[d->path_c[p]];
    const int64_t n = (int64_t)(2 * la + 1) * (2 * lb + 1) * (2 * lc + 1);
    if (capacity < n) return TP_ERR_ARG;
    std::memcpy(out, d->cg[p], sizeof(double) * n);
    return TP_OK;
}

extern "C" void tp_desc_destroy(tp_desc *d) { free_desc(d); }

// ---- symmetric contraction: the basis of symmetric equivariant tensors ------------
//
// For degree nu and output irrep L, the tensors T[i_1..i_nu, k] over the
// components of one channel of the input (i over every block) that are
// symmetric in the nu slots and equivariant. Spanned by the symmetrised
// coupling trees built from this file's Clebsch-Gordan tensors:
//   nu = 1: the identity on each block of type L;
//   nu = 2: C^{l1 l2 L} on blocks (b1, b2) with p1 p2 = pL;
//   nu = 3: sum_m C^{l1 l2 l12}[i1,i2,m] C^{l12 l3 L}[m,i3,k] for every
//           intermediate l12, with p1 p2 p3 = pL;
// each symmetrised over the orderings of its slots. The span is then made
// canonical: reduced row echelon form of the flattened candidates (row-major
// over (i_1..i_nu, k)), each row scaled to unit norm, leading entry positive.

struct tp_symc {
    int mul, n_in, n_out, max_degree;
    int in_l[8], in_p[8], in_off[8];   // per channel: component offsets (mul 1)
    int out_l[8], out_p[8], out_off[8];  // output blocks (element offsets, ir_mul)
    int D, dim_in, dim_out;
    int n_terms;
    int term_nu[32], term_c[32], term_nq[32], term_q0[32];
    std::vector<double> basis[32];     // [nq][D^nu][2L+1]
    int n_weights;
    int num_paths[3], weights_per_degree[3];
    std::vector<tpc::SymcEntry> entries;  // the kernel's table
};

namespace {
bool build_symc_entries(tp_symc *s);
}  // namespace

namespace {

void symmetrise(std::vector<double> &T, int D, int nu, int K) {
    if (nu == 1) return;
    std::vector<double> S(T.size(), 0.0);
    if (nu == 2) {
        for (int a = 0; a < D; ++a)
            for (int b = 0; b < D; ++b)
                for (int k = 0; k < K; ++k) S[(a * D + b) * K + k] = T[(a * D + b) * K + k] + T[(b * D + a) * K + k];
    } else {
        const int perm[6][3] = {{0, 1, 2}, {0, 2, 1}, {1, 0, 2}, {1, 2, 0}, {2, 0, 1}, {2, 1, 0}};
        for (int a = 0; a < D; ++a)
            for (int b = 0; b < D; ++b)
                for (int c = 0; c < D; ++c) {
                    const int idx[3] = {a, b, c};
                    for (int k = 0; k < K; ++k) {
                        double v = 0.0;
                        for (int q = 0; q < 6; ++q)
                            v += T[((idx[perm[q][0]] * D + idx[perm[q][1]]) * D + idx[perm[q][2]]) * K + k];
                        S[((a * D + b) * D + c) * K + k] = v;
                    }
                }
    }
    T.swap(S);
}

// rows (each of length n) -> canonical basis of their span
std::vector<std::vector<double>> rref_canonical(std::vector<std::vector<double>> A, size_t n) {
    size_t r = 0;
    for (size_t c = 0; c < n && r < A.size(); ++c) {
        size_t piv = r;
        for (size_t q = r; q < A.size(); ++q)
            if (std::fabs(A[q][c]) > std::fabs(A[piv][c])) piv = q;
        if (std::fabs(A[piv][c]) < 1e-9) continue;
        std::swap(A[r], A[piv]);
        const double inv = 1.0 / A[r][c];
        for (size_t j = 0; j < n; ++j) A[r][j] *= inv;
        for (size_t q = 0; q < A.size(); ++q) {
            if (q == r || A[q][c] == 0.0) continue;
            const double f = A[q][c];
            for (size_t j = 0; j < n; ++j) A[q][j] -= f * A[r][j];
        }
        ++r;
    }
    A.resize(r);
    for (auto &row : A) {
        double nrm = 0.0, lead = 0.0;
        for (double &v : row) {
            if (std::fabs(v) < 1e-12) v = 0.0;
            nrm += v * v;
            if (lead == 0.0 && std::fabs(v) > 1e-9) lead = v;
        }
        const double s = (lead < 0 ? -1.0 : 1.0) / std::sqrt(nrm);
        for (double &v : row) v *= s;
    }
    return A;
}

}  // namespace

extern "C" tp_status tp_symc_create(const char *irreps_in, const char *irreps_out, int32_t max_degree,
                                    tp_symc **out) {
    if (!irreps_in || !irreps_out || !out || max_degree < 1) return TP_ERR_ARG;
    *out = nullptr;
    if (max_degree > 3) return TP_ERR_UNSUPPORTED;
    std::vector<Term> tin, tout;
    if (!parse_irreps(irreps_in, tin) || !parse_irreps(irreps_out, tout)) return TP_ERR_PARSE;
    if ((tin[0].p != 0) != (tout[0].p != 0)) return TP_ERR_PARSE;
    if (tin.size() > 8 || tout.size() > 8) return TP_ERR_UNSUPPORTED;
    tp_symc *s = new (std::nothrow) tp_symc();
    if (!s) return TP_ERR_ARG;
    s->mul = tin[0].mul;
    s->max_degree = max_degree;
    s->n_in = (int)tin.size();
    s->n_out = (int)tout.size();
    int D = 0, off = 0;
    for (int b = 0; b < s->n_in; ++b) {
        if (tin[b].mul != s->mul || tin[b].l > 2) { delete s; return TP_ERR_UNSUPPORTED; }
        s->in_l[b] = tin[b].l; s->in_p[b] = tin[b].p; s->in_off[b] = D;
        D += 2 * tin[b].l + 1;
    }
    for (int c = 0; c < s->n_out; ++c) {
        if (tout[c].mul != s->mul || tout[c].l > 3) { delete s; return TP_ERR_UNSUPPORTED; }
        s->out_l[c] = tout[c].l; s->out_p[c] = tout[c].p; s->out_off[c] = off;
        off += s->mul * (2 * tout[c].l + 1);
    }
    if (s->mul % 32 != 0) { delete s; return TP_ERR_UNSUPPORTED; }
    s->D = D;
    s->dim_in = D * s->mul;
    s->dim_out = off;
    auto par_ok = [](int p, int q) { return p == 0 || p == q; };
    s->n_terms = 0;
    s->n_weights = 0;
    for (int nu = 1; nu <= max_degree; ++nu) {
        s->num_paths[nu - 1] = s->weights_per_degree[nu - 1] = 0;
        for (int c = 0; c < s->n_out; ++c) {
            const int L = s->out_l[c], pL = s->out_p[c], K = 2 * L + 1;
            size_t n = (size_t)K;
            for (int t = 0; t < nu; ++t) n *= (size_t)D;
            std::vector<std::vector<double>> cand;
            auto at3 = [&](int a, int b, int cc, int k) { return (((size_t)a * D + b) * D + cc) * K + k; };
            if (nu == 1) {
                for (int b = 0; b < s->n_in; ++b) {
                    if (s->in_l[b] != L || !par_ok(s->in_p[b], pL)) continue;
                    std::vector<double> T(n, 0.0);
                    for (int k = 0; k < K; ++k) T[(size_t)(s->in_off[b] + k) * K + k] = 1.0;
                    cand.push_back(T);
                }
            } else if (nu == 2) {
                for (int b1 = 0; b1 < s->n_in; ++b1)
                    for (int b2 = 0; b2 < s->n_in; ++b2) {
                        const int l1 = s->in_l[b1], l2 = s->in_l[b2];
                        if (L < std::abs(l1 - l2) || L > l1 + l2 || !par_ok(s->in_p[b1] * s->in_p[b2], pL)) continue;
                        std::vector<double> C((size_t)(2 * l1 + 1) * (2 * l2 + 1) * K);
                        real_cg(l1, l2, L, C.data());
                        std::vector<double> T(n, 0.0);
                        for (int i = 0; i < 2 * l1 + 1; ++i)
                            for (int j = 0; j < 2 * l2 + 1; ++j)
                                for (int k = 0; k < K; ++k)
                                    T[((size_t)(s->in_off[b1] + i) * D + s->in_off[b2] + j) * K + k] =
                                        C[((size_t)i * (2 * l2 + 1) + j) * K + k];
                        symmetrise(T, D, 2, K);
                        cand.push_back(T);
                    }
            } else {
                for (int b1 = 0; b1 < s->n_in; ++b1)
                    for (int b2 = 0; b2 < s->n_in; ++b2)
                        for (int b3 = 0; b3 < s->n_in; ++b3) {
                            const int l1 = s->in_l[b1], l2 = s->in_l[b2], l3 = s->in_l[b3];
                            if (!par_ok(s->in_p[b1] * s->in_p[b2] * s->in_p[b3], pL)) continue;
                            for (int l12 = std::abs(l1 - l2); l12 <= l1 + l2; ++l12) {
                                if (L < std::abs(l12 - l3) || L > l12 + l3) continue;
                                const int n12 = 2 * l12 + 1;
                                std::vector<double> C1((size_t)(2 * l1 + 1) * (2 * l2 + 1) * n12),
                                    C2((size_t)n12 * (2 * l3 + 1) * K);
                                real_cg(l1, l2, l12, C1.data());
                                real_cg(l12, l3, L, C2.data());
                                std::vector<double> T(n, 0.0);
                                for (int i = 0; i < 2 * l1 + 1; ++i)
                                    for (int j = 0; j < 2 * l2 + 1; ++j)
                                        for (int q = 0; q < 2 * l3 + 1; ++q)
                                            for (int k = 0; k < K; ++k) {
                                                double v = 0.0;
                                                for (int m = 0; m < n12; ++m)
                                                    v += C1[((size_t)i * (2 * l2 + 1) + j) * n12 + m] *
                                                         C2[((size_t)m * (2 * l3 + 1) + q) * K + k];
                                                T[at3(s->in_off[b1] + i, s->in_off[b2] + j, s->in_off[b3] + q, k)] = v;
                                            }
                                symmetrise(T, D, 3, K);
                                cand.push_back(T);
                            }
                        }
            }
            std::vector<std::vector<double>> B = rref_canonical(cand, n);
            if (B.empty()) continue;
            if (s->n_terms >= 32) { delete s; return TP_ERR_UNSUPPORTED; }
            const int t = s->n_terms++;
            s->term_nu[t] = nu;
            s->term_c[t] = c;
            s->term_nq[t] = (int)B.size();
            s->term_q0[t] = s->n_weights;
            s->n_weights += (int)B.size();
            s->weights_per_degree[nu - 1] += (int)B.size();
            s->basis[t].assign(B.size() * n, 0.0);
            for (size_t q = 0; q < B.size(); ++q)
                for (size_t j = 0; j < n; ++j) {
                    s->basis[t][q * n + j] = B[q][j];
                    if (B[q][j] != 0.0) ++s->num_paths[nu - 1];
                }
        }
    }
    if (s->n_terms == 0 || !build_symc_entries(s)) { delete s; return TP_ERR_UNSUPPORTED; }
    *out = s;
    return TP_OK;
}

extern "C" tp_status tp_symc_query(const tp_symc *s, tp_symc_info *info) {
    if (!s || !info) return TP_ERR_ARG;
    info->mul = s->mul;
    info->dim_in = s->dim_in;
    info->dim_out = s->dim_out;
    info->max_degree = s->max_degree;
    info->n_weights = s->n_weights;
    info->n_terms = s->n_terms;
    for (int k = 0; k < 3; ++k) {
        info->num_paths[k] = k < s->max_degree ? s->num_paths[k] : 0;
        info->weights_per_degree[k] = k < s->max_degree ? s->weights_per_degree[k] : 0;
    }
    return TP_OK;
}

extern "C" tp_status tp_symc_term(const tp_symc *s, int32_t t, int32_t *nu, int32_t *out_block, int32_t *n_q,
                                  double *basis, int64_t capacity) {
    if (!s || t < 0 || t >= s->n_terms || !nu || !out_block || !n_q) return TP_ERR_ARG;
    *nu = s->term_nu[t];
    *out_block = s->term_c[t];
    *n_q = s->term_nq[t];
    if (basis) {
        if (capacity < (int64_t)s->basis[t].size()) return TP_ERR_ARG;
        std::memcpy(basis, s->basis[t].data(), sizeof(double) * s->basis[t].size());
    }
    return TP_OK;
}

extern "C" void tp_symc_destroy(tp_symc *s) { delete s; }

namespace {
// The nonzero basis entries in weight order (the kernel's table).
bool build_symc_entries(tp_symc *s) {
    s->entries.clear();
    for (int t = 0; t < s->n_terms; ++t) {
        const int nu = s->term_nu[t], c = s->term_c[t], K = 2 * s->out_l[c] + 1, D = s->D;
        size_t per = (size_t)K;
        for (int q = 0; q < nu; ++q) per *= (size_t)D;
        for (int q = 0; q < s->term_nq[t]; ++q)
            for (size_t j = 0; j < per; ++j) {
                const double v = s->basis[t][q * per + j];
                if (v == 0.0) continue;
                if ((int)s->entries.size() >= tpc::kSymcMaxEntries) return false;
                size_t r = j;
                const int k = (int)(r % K);
                r /= K;
                int idx[3] = {0, 0, 0};
                for (int a = nu - 1; a >= 0; --a) {
                    idx[a] = (int)(r % D);
                    r /= D;
                }
                tpc::SymcEntry e;
                e.nu = (uint8_t)nu;
                e.i1 = (uint8_t)idx[0];
                e.i2 = (uint8_t)idx[1];
                e.i3 = (uint8_t)idx[2];
                e.row = (uint16_t)(s->out_off[c] / s->mul + k);
                e.q = (uint16_t)(s->term_q0[t] + q);
                e.coef = (float)v;
                s->entries.push_back(e);
            }
    }
    // grouped by output row (then weight, then position), the order the kernel sums in
    std::stable_sort(s->entries.begin(), s->entries.end(), [](const tpc::SymcEntry &a, const tpc::SymcEntry &b) {
        return a.row != b.row ? a.row < b.row : a.q < b.q;
    });
    return true;
}
}  // namespace

namespace tpc {
const SymcEntry *symc_table(const tp_symc *s, int *n) {
    *n = (int)s->entries.size();
    return s->entries.data();
}
int symc_mul(const tp_symc *s) { return s->mul; }
int symc_D(const tp_symc *s) { return s->D; }
int symc_rows_out(const tp_symc *s) { return s->dim_out / s->mul; }
int symc_n_weights(const tp_symc *s) { return s->n_weights; }
}  // namespace tpc
