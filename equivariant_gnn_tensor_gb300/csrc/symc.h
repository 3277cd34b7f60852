// Kernel table of a symmetric contraction (shared by the host builder and the kernel).
#pragma once
#include <cstdint>

struct tp_symc;

namespace tpc {

// One nonzero basis entry: coef * prod_{t < nu} b[i_t] adds to output row
// `row` (an ir_mul row of mul channels) with weight q.
struct SymcEntry {
    uint8_t nu, i1, i2, i3;
    uint16_t row;
    uint16_t q;
    float coef;
};

constexpr int kSymcMaxEntries = 2000;

// The entries of a descriptor (grouped by output row), its multiplicity, number of
// input components per channel, output rows and weights per element and channel.
const SymcEntry *symc_table(const tp_symc *s, int *n);
int symc_mul(const tp_symc *s);
int symc_D(const tp_symc *s);
int symc_rows_out(const tp_symc *s);
int symc_n_weights(const tp_symc *s);

}  // namespace tpc
