// Compile-time path programs (host and device).
//
// A program fixes, at compile time, the list of channelwise paths
// (l_a, l_b, l_c) of one irreps shape and, for each path, which entries
// (i, k) of the per-edge matrix M_p[i][k] = sum_j C_p[i,j,k] sh[b_p, j] can be
// nonzero. Kernels instantiated for a program run each edge as straight-line
// code over its paths and touch only those entries; the host builds the
// runtime tables for the same layout and uses such a kernel only after
// checking that every nonzero Clebsch-Gordan entry falls inside the pattern.
//
// Pattern rule (real basis, m = i - l, cos-type for m >= 0, sin-type for
// m < 0): a product of harmonics of orders m1 and m2 only reaches orders with
// |m3| = |m1| + |m2| or ||m1| - |m2||, and it is sin-type exactly when one of
// the factors is; for l_a + l_b + l_c odd the coupling exchanges the two types.
// Programs used here: "natural parity" shapes, input degrees 0..LI, harmonic
// degrees 0..LSH, output degrees 0..LO, parities (-1)^l, so a path exists
// when |la - lb| <= lc <= min(la + lb, LO) and la + lb + lc is even.
#pragma once

namespace tpc {

constexpr int kProgMaxPaths = 32;
constexpr int kProgMaxNz = 49;

struct ProgPath {
    int la, lb, lc;
};

struct Program {
    int n;                                      // paths
    ProgPath p[kProgMaxPaths];
    int nz[kProgMaxPaths];                      // pattern entries of path t
    int moff[kProgMaxPaths];                    // offset of path t in M (floats, multiple of 4)
    int R;                                      // M floats per edge (padded)
    unsigned char ik[kProgMaxPaths][kProgMaxNz];  // entry q of path t: i*8 + k
};

constexpr int pabs(int v) { return v < 0 ? -v : v; }

constexpr bool m_entry_possible(int la, int lb, int lc, int i, int k) {
    const int m1 = i - la, m3 = k - lc;
    const bool odd = ((la + lb + lc) & 1) != 0;
    for (int m2 = -lb; m2 <= lb; ++m2) {
        const int a = pabs(m1), b = pabs(m2), c = pabs(m3);
        if (!(c == a + b || c == pabs(a - b))) continue;
        bool sin_prod = (m1 < 0) != (m2 < 0);
        if (odd) sin_prod = !sin_prod;
        if (sin_prod != (m3 < 0)) continue;
        return true;
    }
    return false;
}

// The harmonic components j (0..2lb, ascending) that can couple input row i
// to output row k of path (la, lb, lc) under the same rule: at most two, one
// per value of |m2|; `slot` 0 or 1, -1 when there is no such component.
constexpr int m_entry_j(int la, int lb, int lc, int i, int k, int slot) {
    const int m1 = i - la, m3 = k - lc;
    const bool odd = ((la + lb + lc) & 1) != 0;
    int found = 0;
    for (int m2 = -lb; m2 <= lb; ++m2) {
        const int a = pabs(m1), b = pabs(m2), c = pabs(m3);
        if (!(c == a + b || c == pabs(a - b))) continue;
        bool sin_prod = (m1 < 0) != (m2 < 0);
        if (odd) sin_prod = !sin_prod;
        if (sin_prod != (m3 < 0)) continue;
        if (found == slot) return m2 + lb;
        ++found;
    }
    return -1;
}

constexpr Program make_natural_program(int LI, int LSH, int LO) {
    Program P{};
    P.n = 0;
    for (int la = 0; la <= LI; ++la)
        for (int lb = 0; lb <= LSH; ++lb)
            for (int lc = pabs(la - lb); lc <= la + lb; ++lc) {
                if (lc > LO || ((la + lb + lc) & 1)) continue;
                P.p[P.n] = ProgPath{la, lb, lc};
                ++P.n;
            }
    int off = 0;
    for (int t = 0; t < P.n; ++t) {
        const int la = P.p[t].la, lb = P.p[t].lb, lc = P.p[t].lc;
        int q = 0;
        for (int i = 0; i < 2 * la + 1; ++i)
            for (int k = 0; k < 2 * lc + 1; ++k)
                if (m_entry_possible(la, lb, lc, i, k)) {
                    P.ik[t][q] = (unsigned char)(i * 8 + k);
                    ++q;
                }
        P.nz[t] = q;
        P.moff[t] = off;
        off += (q + 3) / 4 * 4;
    }
    P.R = off;
    return P;
}

// Shapes that have compiled programs: (LI, LSH, LO).
struct ProgShape {
    int li, lsh, lo;
};
constexpr ProgShape kProgShapes[] = {{1, 1, 1}, {1, 2, 2}, {2, 3, 2}, {3, 3, 3}};
constexpr int kNumProgShapes = 4;

template <int LI, int LSH, int LO>
struct NaturalProgram {
    static constexpr Program P = make_natural_program(LI, LSH, LO);
};

}  // namespace tpc
