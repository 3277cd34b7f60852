// Stable counting sort of int32 keys in [0, N) -> (perm, row_ptr, sorted keys),
// the destination-sorted CSR the convolution streams ("cuEquivariance in
// PyTorch", Limitations and backends: indexed kernels need sorted indices;
// SegmentedPolynomial: gather and scatter: int32 index tensors on the device).
//
// LSD radix sort over ceil(log2 N) key bits, up to 8 bits per pass. Each pass:
//   hist    - one block per tile of 2048 keys counts its digits;
//   scan    - one block turns the digit-major [digit][tile] counts into
//             exclusive offsets;
//   scatter - each warp of a tile ranks its 256 keys in input order
//             (__match_any_sync peers + per-warp running counters), so equal
//             digits keep their order across warps, tiles and passes.
// row_ptr[d] is then the lower bound of d in the sorted keys. Integer work
// only: the result is exact and deterministic.
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>

#include "../../include/tpconv.h"
#include "common.cuh"

namespace tpc {

constexpr int kTile = 2048;
constexpr int kSortThreads = 256;

__global__ void radix_hist_kernel(const int32_t *__restrict__ keys, int64_t E, int shift, int nbits,
                                  int32_t *__restrict__ tile_hist, int n_tiles, int32_t N, int check,
                                  int *status) {
    __shared__ int32_t hist[256];
    const int nb = 1 << nbits;
    for (int d = threadIdx.x; d < nb; d += blockDim.x) hist[d] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kTile;
    bool bad = false;
    for (int q = threadIdx.x; q < kTile; q += blockDim.x) {
        const int64_t idx = base + q;
        if (idx < E) {
            const int32_t k = keys[idx];
            if (check && (k < 0 || k >= N)) bad = true;
            atomicAdd(&hist[((uint32_t)k >> shift) & (nb - 1)], 1);
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, TP_DEV_ERR_INDEX);
    __syncthreads();
    for (int d = threadIdx.x; d < nb; d += blockDim.x) tile_hist[(int64_t)d * n_tiles + blockIdx.x] = hist[d];
}

// Exclusive scan of n int32 counts in place by one block of 1024 threads.
__global__ void exclusive_scan_kernel(int32_t *__restrict__ a, int64_t n) {
    __shared__ int64_t part[1024];
    const int t = threadIdx.x;
    const int64_t per = (n + blockDim.x - 1) / blockDim.x;
    const int64_t lo = min(n, (int64_t)t * per), hi = min(n, lo + per);
    int64_t s = 0;
    for (int64_t i = lo; i < hi; ++i) s += a[i];
    part[t] = s;
    __syncthreads();
    for (int off = 1; off < (int)blockDim.x; off <<= 1) {
        int64_t v = t >= off ? part[t - off] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int64_t run = part[t] - s;
    for (int64_t i = lo; i < hi; ++i) {
        const int32_t v = a[i];
        a[i] = (int32_t)run;
        run += v;
    }
}

__global__ void radix_scatter_kernel(const int32_t *__restrict__ keys_in, const int32_t *__restrict__ vals_in,
                                     int64_t E, int shift, int nbits, const int32_t *__restrict__ tile_off,
                                     int n_tiles, int32_t *__restrict__ keys_out, int32_t *__restrict__ vals_out) {
    constexpr int kWarps = kSortThreads / 32;
    constexpr int kPerWarp = kTile / kWarps;
    __shared__ int32_t whist[kWarps][256];
    const int nb = 1 << nbits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int d = lane; d < nb; d += 32) whist[warp][d] = 0;
    __syncwarp();
    const int64_t wbase = (int64_t)blockIdx.x * kTile + warp * kPerWarp;
    for (int r = 0; r < kPerWarp; r += 32) {
        const int64_t idx = wbase + r + lane;
        if (idx < E) atomicAdd(&whist[warp][((uint32_t)keys_in[idx] >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // base[w][d] = tile offset of d + counts of d in earlier warps of this tile
    for (int d = threadIdx.x; d < nb; d += blockDim.x) {
        int32_t run = tile_off[(int64_t)d * n_tiles + blockIdx.x];
        for (int w = 0; w < kWarps; ++w) {
            const int32_t c = whist[w][d];
            whist[w][d] = run;
            run += c;
        }
    }
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
    for (int r = 0; r < kPerWarp; r += 32) {
        const int64_t idx = wbase + r + lane;
        const bool valid = idx < E;
        int32_t k = 0, v = 0;
        if (valid) {
            k = keys_in[idx];
            v = vals_in ? vals_in[idx] : (int32_t)idx;
        }
        const int d = valid ? (int)(((uint32_t)k >> shift) & (nb - 1)) : 256 + lane;  // invalid lanes match only themselves
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        int32_t pos = 0;
        if (valid) pos = whist[warp][d] + __popc(peers & lt);
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) whist[warp][d] += __popc(peers);
        __syncwarp();
        if (valid) {
            keys_out[pos] = k;
            vals_out[pos] = v;
        }
    }
}

// row_ptr[d] = number of sorted keys < d, for d in [0, N].
__global__ void row_ptr_kernel(const int32_t *__restrict__ sorted, int64_t E, int32_t N, int32_t *__restrict__ row_ptr) {
    const int64_t d = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (d > N) return;
    int64_t lo = 0, hi = E;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)sorted[mid] < d) lo = mid + 1;
        else hi = mid;
    }
    row_ptr[d] = (int32_t)lo;
}

__global__ void copy_i32_kernel(const int32_t *__restrict__ a, int32_t *__restrict__ b, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        b[i] = a[i];
}

static int key_bits(int32_t N) {
    int b = 0;
    while (b < 31 && ((int64_t)1 << b) < (int64_t)N) ++b;
    return b;
}

struct CsrWs {
    size_t tmp_k, tmp_v, fin_k, hist, total;
};

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

static CsrWs csr_ws_layout(int64_t E, int32_t N) {
    (void)N;
    const int64_t n_tiles = (E + kTile - 1) / kTile;
    CsrWs w;
    w.tmp_k = 0;
    w.tmp_v = align256(w.tmp_k + sizeof(int32_t) * (size_t)E);
    w.fin_k = align256(w.tmp_v + sizeof(int32_t) * (size_t)E);
    w.hist = align256(w.fin_k + sizeof(int32_t) * (size_t)E);
    w.total = align256(w.hist + sizeof(int32_t) * (size_t)(256 * (n_tiles > 0 ? n_tiles : 1)));
    return w;
}

size_t csr_workspace_bytes(int64_t E, int32_t N) { return csr_ws_layout(E, N).total; }

// Runs the sort with scratch at `ws` (at least csr_workspace_bytes, 256-aligned).
cudaError_t csr_build_launch(const int32_t *keys, int64_t E, int32_t N, int32_t *perm, int32_t *row_ptr,
                             int32_t *keys_sorted, void *ws, int *status, cudaStream_t stream) {
    const CsrWs L = csr_ws_layout(E, N);
    unsigned char *base = static_cast<unsigned char *>(ws);
    int32_t *tmp_k = reinterpret_cast<int32_t *>(base + L.tmp_k);
    int32_t *tmp_v = reinterpret_cast<int32_t *>(base + L.tmp_v);
    int32_t *fin_k = keys_sorted ? keys_sorted : reinterpret_cast<int32_t *>(base + L.fin_k);
    int32_t *hist = reinterpret_cast<int32_t *>(base + L.hist);
    if (E > 0) {
        const int bits = key_bits(N);
        const int passes = bits == 0 ? 1 : (bits + 7) / 8;
        const int per = bits == 0 ? 1 : (bits + passes - 1) / passes;
        const int n_tiles = (int)((E + kTile - 1) / kTile);
        for (int ps = 0; ps < passes; ++ps) {
            const int shift = ps * per;
            const int nbits = bits == 0 ? 1 : (shift + per <= bits ? per : bits - shift);
            const int32_t *kin = ps == 0 ? keys : (((passes - ps) % 2 == 0) ? fin_k : tmp_k);
            const int32_t *vin = ps == 0 ? nullptr : (((passes - ps) % 2 == 0) ? perm : tmp_v);
            const bool to_final = ((passes - 1 - ps) % 2) == 0;
            int32_t *kout = to_final ? fin_k : tmp_k;
            int32_t *vout = to_final ? perm : tmp_v;
            radix_hist_kernel<<<n_tiles, kSortThreads, 0, stream>>>(kin, E, shift, nbits, hist, n_tiles, N, ps == 0,
                                                                    status);
            exclusive_scan_kernel<<<1, 1024, 0, stream>>>(hist, (int64_t)n_tiles << nbits);
            radix_scatter_kernel<<<n_tiles, kSortThreads, 0, stream>>>(kin, vin, E, shift, nbits, hist, n_tiles,
                                                                       kout, vout);
        }
    }
    row_ptr_kernel<<<(int)((N + 1 + 255) / 256), 256, 0, stream>>>(fin_k, E, N, row_ptr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the sort's scratch lives in this fixed device array
// instead of caller memory. Sized for kNoAllocMaxEdges keys (any N): three
// int32 arrays of that length plus the per-tile digit counts.
constexpr int64_t kNoAllocMaxEdges = int64_t(1) << 18;
constexpr size_t kNoAllocBytes =
    (sizeof(int32_t) * kNoAllocMaxEdges + 255) / 256 * 256 * 3 +
    (sizeof(int32_t) * 256 * ((kNoAllocMaxEdges + kTile - 1) / kTile) + 255) / 256 * 256;
static __device__ __align__(256) unsigned char g_csr_scratch[kNoAllocBytes];

int64_t csr_noalloc_max_edges() { return kNoAllocMaxEdges; }

// Device address of g_csr_scratch on the current device, looked up once per
// device (the name is only a host-side stand-in for the symbol).
cudaError_t csr_noalloc_scratch(void **ptr) {
    static std::mutex mu;
    static std::map<int, void *> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) {
        *ptr = it->second;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_csr_scratch);
    if (e != cudaSuccess) return e;
    if (csr_workspace_bytes(kNoAllocMaxEdges, 1) > kNoAllocBytes) return cudaErrorInvalidValue;
    addr[dev] = p;
    *ptr = p;
    return cudaSuccess;
}

}  // namespace tpc
