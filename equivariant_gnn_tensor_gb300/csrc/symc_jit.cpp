// Symmetric contraction specialised per descriptor: the host writes a CUDA
// kernel whose body is the descriptor's basis as straight-line code, compiles
// it once per device with NVRTC for sm_103a and launches it through the driver
// API. Compared with the table kernel (symc.cu), every node's components sit
// in registers and every entry is one fused multiply-add with its coefficient
// as an immediate operand, so the kernel issues a few instructions per entry
// instead of decoding a table entry and loading its operands.
//
// Generated kernel: one thread per (node, channel), blocks of NPB nodes x mul
// channels (NPB = 256 / mul, at least 1), a grid-stride loop over nodes.
// Per thread: the D components b_i of its channel (coalesced across the
// channel threads), the node's element and its n_weights weights a_q; the
// monomials b_i b_j and b_i b_j b_k the basis needs, each formed once; then per
// output row r, per weight q: u_rq = sum over the (r, q) entries of
// coef * monomial (entries that differ only in the order of their indices are
// merged into one monomial with the summed coefficient), summed pairwise when
// long; out_r = sum_q a_q u_rq with compensated (Kahan) summation. An element
// index out of range sets TP_DEV_ERR_INDEX and gives the node zero rows.
//
// NVRTC is loaded at run time (dlopen); when it or the driver entry points are
// missing, or compilation fails, the caller uses the table kernel instead.
#include <cuda.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <array>
#include <cinttypes>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/tpconv.h"
#include "symc.h"
#include "tables.h"

namespace tpc {
namespace {

// ---- NVRTC, loaded at run time ------------------------------------------------
typedef int nvrtcResult_t;
typedef struct _nvrtcProgram *nvrtcProgram_t;
struct Nvrtc {
    nvrtcResult_t (*create)(nvrtcProgram_t *, const char *, const char *, int, const char *const *,
                            const char *const *) = nullptr;
    nvrtcResult_t (*compile)(nvrtcProgram_t, int, const char *const *) = nullptr;
    nvrtcResult_t (*cubin_size)(nvrtcProgram_t, size_t *) = nullptr;
    nvrtcResult_t (*cubin)(nvrtcProgram_t, char *) = nullptr;
    nvrtcResult_t (*destroy)(nvrtcProgram_t *) = nullptr;
    bool ok = false;
};

const Nvrtc &nvrtc() {
    static Nvrtc n;
    static std::once_flag once;
    std::call_once(once, [] {
        void *h = nullptr;
        for (const char *name : {"libnvrtc.so.13", "libnvrtc.so", "/usr/local/cuda/lib64/libnvrtc.so.13"}) {
            h = dlopen(name, RTLD_NOW | RTLD_LOCAL);
            if (h) break;
        }
        if (!h) return;
        n.create = reinterpret_cast<decltype(n.create)>(dlsym(h, "nvrtcCreateProgram"));
        n.compile = reinterpret_cast<decltype(n.compile)>(dlsym(h, "nvrtcCompileProgram"));
        n.cubin_size = reinterpret_cast<decltype(n.cubin_size)>(dlsym(h, "nvrtcGetCUBINSize"));
        n.cubin = reinterpret_cast<decltype(n.cubin)>(dlsym(h, "nvrtcGetCUBIN"));
        n.destroy = reinterpret_cast<decltype(n.destroy)>(dlsym(h, "nvrtcDestroyProgram"));
        n.ok = n.create && n.compile && n.cubin_size && n.cubin && n.destroy;
    });
    return n;
}

// ---- driver entry points --------------------------------------------------------
struct Driver {
    CUresult (*load)(CUmodule *, const void *) = nullptr;
    CUresult (*get)(CUfunction *, CUmodule, const char *) = nullptr;
    CUresult (*launch)(CUfunction, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, CUstream,
                       void **, void **) = nullptr;
    bool ok = false;
};

const Driver &driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        auto get = [](const char *sym, void **p) {
            cudaDriverEntryPointQueryResult q;
            return cudaGetDriverEntryPointByVersion(sym, p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess;
        };
        void *a = nullptr, *b = nullptr, *c = nullptr;
        if (get("cuModuleLoadData", &a) && get("cuModuleGetFunction", &b) && get("cuLaunchKernel", &c)) {
            d.load = reinterpret_cast<decltype(d.load)>(a);
            d.get = reinterpret_cast<decltype(d.get)>(b);
            d.launch = reinterpret_cast<decltype(d.launch)>(c);
            d.ok = true;
        }
    });
    return d;
}

// ---- source generation ----------------------------------------------------------
std::string flit(double v) {  // exact float literal (hexadecimal)
    char buf[64];
    std::snprintf(buf, sizeof(buf), "%af", (double)(float)v);
    return buf;
}

std::string mono_name(const std::array<int, 3> &t, int nu) {
    if (nu == 1) return "b" + std::to_string(t[0]);
    std::string s = "m";
    for (int a = 0; a < nu; ++a) s += "_" + std::to_string(t[a]);
    return s;
}

// Body of the kernel for a descriptor's entries (grouped by row, then weight).
std::string generate(const SymcEntry *tab, int n, int mul, int D, int rows, int nw, int npb) {
    // (row, q) -> sorted monomial -> summed coefficient, in first-seen order
    struct Group {
        int row, q;
        std::vector<std::pair<std::array<int, 3>, int>> keys;  // monomial, nu
        std::vector<double> coef;
    };
    std::vector<Group> groups;
    std::map<std::tuple<int, int, int, int, int>, std::pair<size_t, size_t>> where;
    for (int t = 0; t < n; ++t) {
        const SymcEntry &e = tab[t];
        std::array<int, 3> k = {e.i1, e.nu >= 2 ? e.i2 : -1, e.nu >= 3 ? e.i3 : -1};
        std::sort(k.begin(), k.begin() + e.nu);
        if (groups.empty() || groups.back().row != e.row || groups.back().q != e.q) groups.push_back({e.row, e.q, {}, {}});
        Group &g = groups.back();
        const auto key = std::make_tuple((int)e.row, (int)e.q, k[0], k[1], k[2]);
        auto it = where.find(key);
        if (it != where.end() && it->second.first == groups.size() - 1) {
            g.coef[it->second.second] += e.coef;
        } else {
            where[key] = {groups.size() - 1, g.keys.size()};
            g.keys.push_back({k, (int)e.nu});
            g.coef.push_back(e.coef);
        }
    }
    std::string s;
    const int block = mul * npb, dim_in = D * mul;
    s += "extern \"C\" __global__ void __launch_bounds__(" + std::to_string(block) + ")\n";
    s += "symc_jit(const float *__restrict__ x, const float *__restrict__ wts, const int *__restrict__ element,\n";
    s += "         float *__restrict__ out, int *status, int N, int num_elements) {\n";
    s += "  const int ch = threadIdx.x % " + std::to_string(mul) + ", nb = threadIdx.x / " + std::to_string(mul) + ";\n";
    s += "  for (long long n = (long long)blockIdx.x * " + std::to_string(npb) + " + nb; n < N; n += (long long)gridDim.x * " +
         std::to_string(npb) + ") {\n";
    s += "    const float *xr = x + n * " + std::to_string(dim_in) + " + ch;\n";
    for (int i = 0; i < D; ++i) s += "    const float b" + std::to_string(i) + " = xr[" + std::to_string(i * mul) + "];\n";
    s += "    const int el = element[n];\n";
    s += "    const bool ok = (unsigned)el < (unsigned)num_elements;\n";
    s += "    if (!ok && ch == 0) asm volatile(\"red.global.or.b32 [%0], %1;\" :: \"l\"(status), \"r\"(" +
         std::to_string(TP_DEV_ERR_INDEX) + "));\n";
    s += "    const float *wr = wts + (long long)(ok ? el : 0) * " + std::to_string(nw * mul) + " + ch;\n";
    for (int q = 0; q < nw; ++q) s += "    const float a" + std::to_string(q) + " = wr[" + std::to_string(q * mul) + "];\n";
    // the monomials of degree 2 and 3, each formed once
    std::map<std::string, bool> made;
    for (const Group &g : groups)
        for (const auto &kk : g.keys) {
            const auto &k = kk.first;
            const int nu = kk.second;
            if (nu >= 2) {
                const std::string p = mono_name(k, 2);
                if (!made[p]) {
                    s += "    const float " + p + " = b" + std::to_string(k[0]) + " * b" + std::to_string(k[1]) + ";\n";
                    made[p] = true;
                }
            }
            if (nu == 3) {
                const std::string p = mono_name(k, 3);
                if (!made[p]) {
                    s += "    const float " + p + " = " + mono_name(k, 2) + " * b" + std::to_string(k[2]) + ";\n";
                    made[p] = true;
                }
            }
        }
    s += "    float *orow = out + n * " + std::to_string(rows * mul) + " + ch;\n";
    size_t gi = 0;
    int tmp = 0;
    for (int r = 0; r < rows; ++r) {
        s += "    {\n      float s = 0.f, c = 0.f;\n";
        for (; gi < groups.size() && groups[gi].row == r; ++gi) {
            const Group &g = groups[gi];
            // u = sum of coef * monomial: a chain of FMAs when short, pairwise when long
            std::vector<std::string> terms;
            for (size_t t = 0; t < g.keys.size(); ++t) {
                if ((float)g.coef[t] == 0.f) continue;
                terms.push_back(flit(g.coef[t]) + " * " + mono_name(g.keys[t].first, g.keys[t].second));
            }
            if (terms.empty()) continue;
            std::string u;
            if (terms.size() <= 8) {
                u = "u" + std::to_string(tmp++);
                s += "      float " + u + " = " + terms[0] + ";\n";
                for (size_t t = 1; t < terms.size(); ++t) {
                    const size_t star = terms[t].find(" * ");
                    s += "      " + u + " = fmaf(" + terms[t].substr(0, star) + ", " + terms[t].substr(star + 3) + ", " +
                         u + ");\n";
                }
            } else {
                std::vector<std::pair<std::string, int>> stack;  // (variable, level)
                for (const std::string &t : terms) {
                    std::string v = "u" + std::to_string(tmp++);
                    s += "      const float " + v + " = " + t + ";\n";
                    int lvl = 0;
                    while (!stack.empty() && stack.back().second == lvl) {
                        const std::string w = "u" + std::to_string(tmp++);
                        s += "      const float " + w + " = " + stack.back().first + " + " + v + ";\n";
                        stack.pop_back();
                        v = w;
                        ++lvl;
                    }
                    stack.push_back({v, lvl});
                }
                u = stack.back().first;
                for (int k = (int)stack.size() - 2; k >= 0; --k) {
                    const std::string w = "u" + std::to_string(tmp++);
                    s += "      const float " + w + " = " + stack[k].first + " + " + u + ";\n";
                    u = w;
                }
            }
            s += "      { const float y = fmaf(a" + std::to_string(g.q) + ", " + u +
                 ", -c); const float t = s + y; c = (t - s) - y; s = t; }\n";
        }
        s += "      orow[" + std::to_string(r * mul) + "] = ok ? s : 0.f;\n    }\n";
    }
    s += "  }\n}\n";
    return s;
}

// ---- compiled kernels, one per (device, generated source) ------------------------
struct JitKernel {
    CUfunction fn = nullptr;  // null: compilation failed (the caller uses the table kernel)
    int block = 0, npb = 0;
};
std::mutex g_jit_mu;
std::map<std::pair<int, std::string>, JitKernel> g_jit;

JitKernel compile(const std::string &src, int block, int npb, int cc_major, int cc_minor) {
    JitKernel k;
    const Nvrtc &nv = nvrtc();
    const Driver &dr = driver();
    if (!nv.ok || !dr.ok) return k;
    nvrtcProgram_t prog = nullptr;
    if (nv.create(&prog, src.c_str(), "symc_jit.cu", 0, nullptr, nullptr) != 0) return k;
    // the device's own architecture, with its architecture-specific features
    const std::string arch = "--gpu-architecture=sm_" + std::to_string(cc_major) + std::to_string(cc_minor) + "a";
    const char *opts[] = {arch.c_str(), "--std=c++17", "-default-device"};
    std::vector<char> cubin;
    if (nv.compile(prog, 3, opts) == 0) {
        size_t n = 0;
        if (nv.cubin_size(prog, &n) == 0 && n > 0) {
            cubin.resize(n);
            if (nv.cubin(prog, cubin.data()) != 0) cubin.clear();
        }
    }
    nv.destroy(&prog);
    if (cubin.empty()) return k;
    CUmodule mod = nullptr;  // kept for the life of the process: kernels may be in flight
    if (cudaFree(nullptr) != cudaSuccess) return k;  // the runtime's context is current on this thread
    if (dr.load(&mod, cubin.data()) != CUDA_SUCCESS) return k;
    if (dr.get(&k.fn, mod, "symc_jit") != CUDA_SUCCESS) k.fn = nullptr;
    k.block = block;
    k.npb = npb;
    return k;
}

}  // namespace

// Launches the descriptor's specialised kernel; cudaErrorNotSupported when it
// cannot be built here (the caller then uses the table kernel).
cudaError_t symc_jit_launch(const tp_symc *s, const float *x, const float *weights, const int32_t *element, int32_t N,
                            int32_t num_elements, float *out, int dev, int sms, int *status, cudaStream_t stream) {
    const int mul = symc_mul(s);
    if (mul > 1024) return cudaErrorNotSupported;
    const int npb = mul >= 256 ? 1 : 256 / mul;
    int n_entries = 0;
    const SymcEntry *tab = symc_table(s, &n_entries);
    const std::string src = generate(tab, n_entries, mul, symc_D(s), symc_rows_out(s), symc_n_weights(s), npb);
    JitKernel k;
    {
        std::lock_guard<std::mutex> lk(g_jit_mu);
        auto key = std::make_pair(dev, src);
        auto it = g_jit.find(key);
        if (it == g_jit.end()) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return cudaErrorNotSupported;
            it = g_jit.emplace(key, compile(src, mul * npb, npb, major, minor)).first;
        }
        k = it->second;
    }
    if (!k.fn) return cudaErrorNotSupported;
    long long blocks = ((long long)N + k.npb - 1) / k.npb;
    const long long cap = (long long)sms * (2048 / k.block);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    void *args[] = {&x, &weights, &element, &out, &status, &N, &num_elements};
    const CUresult r = driver().launch(k.fn, (unsigned)blocks, 1, 1, (unsigned)k.block, 1, 1, 0,
                                       reinterpret_cast<CUstream>(stream), args, nullptr);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorLaunchFailure;
}

// The generated source of a descriptor's kernel (tests and inspection).
std::string symc_jit_source(const tp_symc *s) {
    const int mul = symc_mul(s);
    const int npb = mul >= 256 ? 1 : 256 / mul;
    int n_entries = 0;
    const SymcEntry *tab = symc_table(s, &n_entries);
    return generate(tab, n_entries, mul, symc_D(s), symc_rows_out(s), symc_n_weights(s), npb);
}

}  // namespace tpc

extern "C" tp_status tp_symc_kernel_source(const tp_symc *symc, char *buf, int64_t capacity, int64_t *length) {
    if (!symc || !length || capacity < 0 || (capacity > 0 && !buf)) return TP_ERR_ARG;
    const std::string src = tpc::symc_jit_source(symc);
    *length = (int64_t)src.size();
    if (capacity > 0) {
        const size_t n = std::min((size_t)capacity, src.size() + 1);
        std::memcpy(buf, src.c_str(), n);
    }
    return TP_OK;
}
