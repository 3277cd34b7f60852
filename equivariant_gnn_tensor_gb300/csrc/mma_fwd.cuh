// Tensor-core forward for bfloat16 inputs (tcgen05, sm_100+ family), the
// channelwise product of a compiled path program (program.h) with mul = 64.
//
// Per edge the contraction factors into a dense product and a scaled sum:
//   T[u, (p, k)] = sum_i x[src, i, u] * Mbig[i, (p, k)]          (tensor cores)
//   out[d, c_p, k, u] += w[e, p, u] * T[u, (p, k)]               (CUDA cores)
// where Mbig[i, (p, k)] = sum_j C_p[i - la_p^2, j, k] sh[e, b_p, j] for the rows
// i of path p's input block (zero elsewhere) is the per-edge matrix M of every
// path side by side (NCOL = sum_p (2 l_c + 1) columns, padded to a multiple of
// 16). The first line is one tcgen05.mma per edge with x (bf16, as loaded) as
// the A operand and Mbig rounded to bf16 as the B operand, accumulated in fp32
// in tensor memory; the second runs in fp32 on the CUDA cores.
//
// Two edges share one M = 128 MMA: rows 0..63 of the accumulator are the 64
// channels of slot A's edge and rows 64..127 those of slot B's, through two
// K = 16 MMAs into the same accumulator whose A operands are [x_A ; 0] and
// [0 ; x_B] (block-diagonal in K) and whose B operands are Mbig_A and Mbig_B.
// Slot A and slot B walk two contiguous pieces of the destination-sorted edge
// list (pieces 2c and 2c+1 of CTA c), so each slot accumulates its own
// destinations' rows in registers and stores every row once; rows cut by a
// piece boundary go through the same head/tail partials and merge kernel as
// the warp-ring forward. No atomics: bitwise reproducible for a launch geometry.
//
// Warp roles (one CTA, 8 warps):
//   warps 0..3  consumers: warp w reads accumulator lanes 32w..32w+31 (tensor
//               memory lane = accumulator row), i.e. slot w/2, channels
//               32(w%2)..+31; scales by w and sums into 16 output rows held in
//               registers; stores rows when a destination ends.
//   warp 4      producer: per edge pair and stage, one 2-D tensor TMA per slot
//               gathers the 16 x 64 bf16 x row into the 128-byte-swizzled
//               MN-major operand layout, 1-D bulk copies bring the weight and
//               harmonic rows.
//   warps 5..6  build Mbig for both slots from the harmonics as a pair of bf16
//               matrices (K-major, no swizzle), Mbig = hi + lo with
//               hi = bf16(Mbig) and lo = bf16(Mbig - hi), so the product keeps
//               about 16 bits of Mbig. Mbig has a ring of its own.
//   warp 7      one lane issues the four MMAs of a pair (x_A Mbig_A hi and lo,
//               x_B Mbig_B hi and lo) into a free accumulator buffer and
//               commits them to two mbarriers (accumulator ready, Mbig stage
//               free); the warp owns the tensor memory.
// Stages: S shared-memory stages of x, w and sh per slot, kMmaMStages stages
// of Mbig, two accumulator buffers in tensor memory. Every wait is bounded; a
// role that gives up sets TP_DEV_ERR_TIMEOUT and lets its own copies or MMAs
// in flight finish before the CTA releases shared and tensor memory.
#pragma once
#include <cuda.h>

#include "ring_fwd.cuh"

namespace tpc {

constexpr int kMmaMul = 64;
constexpr int kMmaConsumerWarps = 4;
constexpr int kMmaBuilderWarps = 2;
constexpr int kMmaIssuerWarp = kMmaConsumerWarps + 1 + kMmaBuilderWarps;
constexpr int kMmaThreads = (kMmaIssuerWarp + 1) * 32;
constexpr int kMmaMStages = 3;  // Mbig ring
constexpr int kMmaMaxEnt = 320;
constexpr int kMmaTmemCols = 256;  // two accumulator buffers of up to 128 columns

struct MmaParams {
    // shared memory layout (byte offsets from the 1024-aligned base)
    int32_t S;                 // stages
    int32_t z0_off, z1_off;    // 2 KB zero atoms before and after the x stages
    int32_t x_off;             // stage s: x_A at x_off + 4096 s, x_B at + 2048
    int32_t m_off;             // Mbig stage m, slot h, part q (0 hi, 1 lo): m_off + (4 m + 2 h + q) mb_bytes
    int32_t w_off;             // stage s: w_A at w_off + 2 s wb_bytes, w_B at + wb_bytes
    int32_t sh_off;            // stage s: sh_A at sh_off + 2 s sh_bytes, sh_B at + sh_bytes
    int32_t bar_off;           // full[S], sfree[S], mready[3], mfree[3], mdone[2], tempty[2], tmem address
    int32_t smem_bytes;
    // Mbig entries: byte offset in the B operand, harmonic indices j0 | j1 << 4,
    // Mbig = c0 * sh[j0] + c1 * sh[j1]
    int32_t n_ent;
    uint16_t ent_off[kMmaMaxEnt];
    uint8_t ent_j[kMmaMaxEnt];
    float ent_c[kMmaMaxEnt][2];
    const void *w;
    const float *sh;
    const int32_t *src;
    const int32_t *row_ptr;
    float *out;
    float *carry;        // [2 n_pieces][dim_out]
    int32_t *carry_dst;  // [2 n_pieces]
    int *status;
    int32_t n_src, n_dst, n_pieces;
    int64_t E;
    uint64_t wait_ns;
};

// ---- tcgen05 / tensor-TMA wrappers ---------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 operands, fp32 accumulator)
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    const uint32_t acc = accumulate ? 1u : 0u;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// One accumulator row per thread (32 lanes per warp) from tensor memory. A
// wait for the loads always names their registers (as outputs, or as in/out
// operands of a separate wait), so no use of them can be scheduled before the
// data is there.
// 64 consecutive 32-bit columns at taddr, issued without waiting;
// tmem_wait64 waits and takes the registers as in/out operands.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait64(uint32_t (&v)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]), "+r"(v[32]), "+r"(v[33]), "+r"(v[34]), "+r"(v[35]), "+r"(v[36]), "+r"(v[37]), "+r"(v[38]), "+r"(v[39]), "+r"(v[40]), "+r"(v[41]), "+r"(v[42]), "+r"(v[43]), "+r"(v[44]), "+r"(v[45]), "+r"(v[46]), "+r"(v[47]), "+r"(v[48]), "+r"(v[49]), "+r"(v[50]), "+r"(v[51]), "+r"(v[52]), "+r"(v[53]), "+r"(v[54]), "+r"(v[55]), "+r"(v[56]), "+r"(v[57]), "+r"(v[58]), "+r"(v[59]), "+r"(v[60]), "+r"(v[61]), "+r"(v[62]), "+r"(v[63]) : : "memory");
}
// 36 consecutive 32-bit columns at taddr:
__device__ __forceinline__ void tmem_ld36_wait(uint32_t taddr, uint32_t (&v)[36]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%36];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%32, %33, %34, %35}, [%37];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35])
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}

// 2-D tiled tensor load global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar,
                                           uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared-memory matrix descriptor of a tcgen05 operand: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1, layout type
// (0: no swizzle, 2: 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, A MN-major, B K-major, N x M.
__host__ __device__ constexpr uint32_t mma_idesc_bf16(int n, int m) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Columns of the per-edge product T: path t occupies [col0(t), col0(t) + 2 lc + 1).
template <int LI, int LSH, int LO>
struct MmaShape {
    static constexpr Program P = NaturalProgram<LI, LSH, LO>::P;
    static constexpr int ncol() {
        int c = 0;
        for (int t = 0; t < P.n; ++t) c += 2 * P.p[t].lc + 1;
        return c;
    }
    static constexpr int col0(int t) {
        int c = 0;
        for (int q = 0; q < t; ++q) c += 2 * P.p[q].lc + 1;
        return c;
    }
    static constexpr int col_path(int c) {
        for (int t = 0; t < P.n; ++t)
            if (c < col0(t) + 2 * P.p[t].lc + 1) return t;
        return -1;
    }
    static constexpr int NCOL = ncol();
    static constexpr int NPAD = (NCOL + 15) / 16 * 16;
    static constexpr int MB_BYTES = NPAD / 8 * 256;  // K = 16 rows: two 8 x 16-byte core matrices per 8 columns
    static constexpr int WNUM = P.n * kMmaMul;
    static constexpr int WB_BYTES = WNUM * 2;
    static constexpr int SHN = rows_upto(LSH);
    static constexpr int SH_BYTES = SHN * 4;
    static constexpr int RO = rows_upto(LO);
    static constexpr int DOUT = RO * kMmaMul;
};

template <int LI, int LSH, int LO>
__global__ void __launch_bounds__(kMmaThreads, 2)
    mma_fwd_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ MmaParams prm) {
    using SH_ = MmaShape<LI, LSH, LO>;
    constexpr Program P = SH_::P;
    static_assert(rows_upto(LI) == 16, "the A operand is the whole 16-row x block");
    static_assert(SH_::NPAD <= 128, "one accumulator buffer holds at most 128 columns");
    constexpr int MB = SH_::MB_BYTES, WB = SH_::WB_BYTES, SHB = SH_::SH_BYTES, RO = SH_::RO, DOUT = SH_::DOUT;
    constexpr uint32_t IDESC = mma_idesc_bf16(SH_::NPAD, 128);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte-swizzled x atoms need 1024-byte aligned addresses
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = prm.S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + prm.bar_off);
    uint64_t *sfree = full + S;
    uint64_t *mready = sfree + S;
    uint64_t *mfree = mready + kMmaMStages;
    uint64_t *mdone = mfree + kMmaMStages;
    uint64_t *tempty = mdone + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);

    // ---- set-up: barriers, static zeros of the operands, tensor memory ----------
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&sfree[s], kMmaConsumerWarps);
        }
        for (int m = 0; m < kMmaMStages; ++m) {
            mbar_init(&mready[m], kMmaBuilderWarps);
            mbar_init(&mfree[m], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&mdone[b], 1);
            mbar_init(&tempty[b], kMmaConsumerWarps);
        }
    }
    {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int o = threadIdx.x * 16; o < 2048; o += blockDim.x * 16) {
            *reinterpret_cast<uint4 *>(smem + prm.z0_off + o) = z;
            *reinterpret_cast<uint4 *>(smem + prm.z1_off + o) = z;
        }
        for (int o = threadIdx.x * 16; o < 4 * kMmaMStages * MB; o += blockDim.x * 16)
            *reinterpret_cast<uint4 *>(smem + prm.m_off + o) = z;
    }
    fence_proxy_async_smem();  // the zeros are read by the tensor cores (async proxy)
    fence_barrier_init();
    if (warp == kMmaIssuerWarp) {
        tmem_alloc(smem_u32(tmem_slot), kMmaTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nP = prm.n_pieces;
    const int E = (int)prm.E;  // launched only for E < 2^31
    auto piece_lo = [&](int p) -> int { return (int)((int64_t)p * E / nP); };
    const int pA = 2 * blockIdx.x, pB = pA + 1;
    const int loA = piece_lo(pA), loB = piece_lo(pB), hiB = piece_lo(pB + 1);
    const int nA = loB - loA, nB = hiB - loB;
    const int npairs = max(nA, nB);
    bool failed = false;

    if (warp < kMmaConsumerWarps) {
        // ================================ consumers ================================
        const int h = warp >> 1;           // slot
        const int u = (warp & 1) * 32 + lane;  // channel
        const int p = pA + h;
        const int lo = h ? loB : loA, hi = h ? hiB : loB, nh = hi - lo;
        const int N = prm.n_dst;
        const int32_t *rp = prm.row_ptr;
        // destinations of this piece (as in the warp-ring kernel)
        const int f0 = warp_first_geq(rp, N, lo, lane);
        const int f1 = warp_first_geq(rp, N, hi, lane);
        const int r0 = rp[min(f0, N)], r1 = rp[min(f1, N)];
        int d_start = min(f0, N);
        const bool earlier = d_start > 0 && r0 > lo;
        if (earlier) d_start -= 1;
        int d_end = f1;
        if (p == nP - 1 || d_end > N) d_end = N;
        if (d_end < d_start) d_end = d_start;
        const int head_dst = (earlier && d_start < d_end) ? d_start : -1;
        int tail_dst = (p < nP - 1 && d_end > d_start && r1 > hi) ? d_end - 1 : -1;
        if (tail_dst == head_dst) tail_dst = -1;
        if ((warp & 1) == 0 && lane == 0) {
            prm.carry_dst[2 * p] = head_dst;
            prm.carry_dst[2 * p + 1] = tail_dst;
        }
        int wbase = d_start;
        int wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
        auto rp_get = [&](int d) -> int {
            if (d < wbase || d >= wbase + 32) {
                wbase = d;
                wv = (wbase + lane <= N) ? rp[wbase + lane] : 0;
            }
            return __shfl_sync(0xffffffffu, wv, d - wbase);
        };
        int cur_d = d_start, seg_end = 0;
        auto enter = [&](int d) {
            if (d >= d_end) return;
            const int a = rp_get(d);
            int b = rp_get(d + 1);
            if (a < 0 || b < a || b > E) {
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_SEGMENT);
                b = a < 0 ? 0 : (a > E ? E : a);
            }
            seg_end = b < hi ? b : hi;
        };
        float acc[RO];
#pragma unroll
        for (int r = 0; r < RO; ++r) acc[r] = 0.f;
        auto store_row = [&](int d) {
            float *orow;
            if (d == head_dst) orow = prm.carry + (int64_t)(2 * p) * DOUT;
            else if (d == tail_dst) orow = prm.carry + (int64_t)(2 * p + 1) * DOUT;
            else orow = prm.out + (int64_t)d * DOUT;
#pragma unroll
            for (int r = 0; r < RO; ++r) {
                orow[r * kMmaMul + u] = acc[r];
                acc[r] = 0.f;
            }
        };
        enter(cur_d);
        const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
        static_assert(SH_::NCOL > 64 && SH_::NCOL <= 100, "T is read as 64 + 36 columns");
        for (int k = 0; k < npairs; ++k) {
            const int b = k & 1, s = k % S;
            const bool live = k < nh;
            if (!__all_sync(0xffffffffu, mbar_wait(&mdone[b], (uint32_t)(k >> 1) & 1u, prm.wait_ns))) {
                failed = true;
                break;
            }
            tc_fence_after();
            const __nv_bfloat16 *wrow =
                reinterpret_cast<const __nv_bfloat16 *>(smem + prm.w_off + (2 * s + h) * WB) + u;
            // out rows += w_t * T[col] for the columns [C0, C0 + NC) held in Tq, in path order
            float wt[P.n];
            auto fma_cols = [&](auto c0c, auto ncc, const auto &Tq) {
                constexpr int C0 = decltype(c0c)::value, NC = decltype(ncc)::value;
                static_for<NC>([&](auto cc) {
                    constexpr int c = C0 + decltype(cc)::value;
                    if constexpr (c < SH_::NCOL) {
                        constexpr int t = SH_::col_path(c), kk = c - SH_::col0(t), LC = P.p[t].lc;
                        acc[LC * LC + kk] = fmaf(wt[t], __uint_as_float(Tq[decltype(cc)::value]), acc[LC * LC + kk]);
                    }
                });
            };
            uint32_t T1[36];
            if (live) {
                // the weight row landed with the stage (the MMA already consumed its x)
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)(k / S) & 1u, prm.wait_ns))) {
                    failed = true;
                    break;
                }
                uint32_t T0[64];
                tmem_ld64(trow + b * 128, T0);  // on its way while w is read and rows are stored
#pragma unroll
                for (int t = 0; t < P.n; ++t) wt[t] = __bfloat162float(wrow[t * kMmaMul]);
                const int e = lo + k;
                while (e >= seg_end && cur_d < d_end) {
                    store_row(cur_d);
                    ++cur_d;
                    enter(cur_d);
                }
                tmem_wait64(T0);
                fma_cols(std::integral_constant<int, 0>{}, std::integral_constant<int, 64>{}, T0);
                tmem_ld36_wait(trow + b * 128 + 64, T1);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tempty[b]);
                mbar_arrive(&sfree[s]);
            }
            if (live) fma_cols(std::integral_constant<int, 64>{}, std::integral_constant<int, 36>{}, T1);
        }
        if (failed) {
            if (lane == 0) {
                set_status(prm.status, TP_DEV_ERR_TIMEOUT);
                if ((warp & 1) == 0) {
                    prm.carry_dst[2 * p] = -1;
                    prm.carry_dst[2 * p + 1] = -1;
                }
            }
        } else {
            while (cur_d < d_end) {
                store_row(cur_d);
                ++cur_d;
                enter(cur_d);
            }
        }
    } else if (warp == kMmaConsumerWarps) {
        // ================================ producer =================================
        const uint64_t pol_keep = policy_evict_last();
        const uint64_t pol_stream = policy_evict_first();
        const unsigned char *wg = static_cast<const unsigned char *>(prm.w);
        const unsigned char *shg = reinterpret_cast<const unsigned char *>(prm.sh);
        // source indices of 32 pairs per register, loaded one batch ahead
        auto load_batch = [&](int k0, int &sa, int &sb) {
            const int k = k0 + lane;
            sa = k < nA ? prm.src[loA + k] : 0;
            sb = k < nB ? prm.src[loB + k] : 0;
        };
        int curA, curB, nxtA, nxtB;
        load_batch(0, curA, curB);
        load_batch(32, nxtA, nxtB);
        int k_issued = 0;
        for (int k = 0; k < npairs; ++k) {
            const int s = k % S;
            if ((k & 31) == 0 && k > 0) {
                curA = nxtA;
                curB = nxtB;
                load_batch(k + 32, nxtA, nxtB);
            }
            const int sa = __shfl_sync(0xffffffffu, curA, k & 31), sb = __shfl_sync(0xffffffffu, curB, k & 31);
            if (!__all_sync(0xffffffffu, mbar_wait(&sfree[s], ((uint32_t)(k / S) & 1u) ^ 1u, prm.wait_ns))) {
                failed = true;
                break;
            }
            const bool liveA = k < nA, liveB = k < nB;
            const bool okA = liveA && (uint32_t)sa < (uint32_t)prm.n_src;
            const bool okB = liveB && (uint32_t)sb < (uint32_t)prm.n_src;
            unsigned char *xa = smem + prm.x_off + s * 4096, *xb = xa + 2048;
            if ((liveA && !okA) || (liveB && !okB)) {
                // an out-of-range source: flag it, and give the edge a zero row
                if (lane == 0) set_status(prm.status, TP_DEV_ERR_INDEX);
                const uint4 z = make_uint4(0, 0, 0, 0);
                for (int o = lane * 16; o < 2048; o += 512) {
                    if (liveA && !okA) *reinterpret_cast<uint4 *>(xa + o) = z;
                    if (liveB && !okB) *reinterpret_cast<uint4 *>(xb + o) = z;
                }
                fence_proxy_async_smem();
            }
            const uint32_t bytes = (liveA ? (uint32_t)(WB + SHB) : 0u) + (liveB ? (uint32_t)(WB + SHB) : 0u) +
                                   (okA ? 2048u : 0u) + (okB ? 2048u : 0u);
            if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
            __syncwarp();
            const int eA = loA + k, eB = loB + k;
            if (lane == 0 && okA) tma_load_2d(xa, &tmap_x, 0, sa * 16, &full[s], pol_keep);
            if (lane == 1 && okB) tma_load_2d(xb, &tmap_x, 0, sb * 16, &full[s], pol_keep);
            if (lane == 2 && liveA)
                bulk_g2s(smem + prm.w_off + (2 * s) * WB, wg + (int64_t)eA * WB, WB, &full[s], pol_stream);
            if (lane == 3 && liveB)
                bulk_g2s(smem + prm.w_off + (2 * s + 1) * WB, wg + (int64_t)eB * WB, WB, &full[s], pol_stream);
            if (lane == 4 && liveA)
                bulk_g2s(smem + prm.sh_off + (2 * s) * SHB, shg + (int64_t)eA * SHB, SHB, &full[s], pol_stream);
            if (lane == 5 && liveB)
                bulk_g2s(smem + prm.sh_off + (2 * s + 1) * SHB, shg + (int64_t)eB * SHB, SHB, &full[s], pol_stream);
            k_issued = k + 1;
        }
        if (failed) {
            if (lane == 0) set_status(prm.status, TP_DEV_ERR_TIMEOUT);
            // let this warp's copies land (full time limit) before shared memory is released
            for (int k = max(0, k_issued - S); k < k_issued; ++k)
                (void)mbar_wait(&full[k % S], (uint32_t)(k / S) & 1u, kWaitNs);
        }
    } else if (warp < kMmaIssuerWarp) {
        // ============================== Mbig builders ==============================
        const int tm = threadIdx.x - (kMmaConsumerWarps + 1) * 32;
        constexpr int NB = kMmaBuilderWarps * 32;
        constexpr int PER = (kMmaMaxEnt + NB - 1) / NB;
        // entries of this thread; a thread with fewer than PER entries writes
        // zeros into a padding column of Mbig (its T column is never read), so
        // the loop below is straight-line code
        constexpr uint32_t kPadOff = (uint32_t)((SH_::NPAD - 1) / 8 * 256 + ((SH_::NPAD - 1) % 8) * 16);
        static_assert(SH_::NPAD > SH_::NCOL, "needs a padding column");
        uint32_t e_off[PER], e_j0[PER], e_j1[PER];
        float e_c0[PER], e_c1[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int r = tm + q * NB;
            const bool ok = r < prm.n_ent;
            e_off[q] = ok ? prm.ent_off[r] : kPadOff;
            e_j0[q] = ok ? (prm.ent_j[r] & 15u) * 4u : 0u;
            e_j1[q] = ok ? (prm.ent_j[r] >> 4) * 4u : 0u;
            e_c0[q] = ok ? prm.ent_c[r][0] : 0.f;
            e_c1[q] = ok ? prm.ent_c[r][1] : 0.f;
        }
        for (int k = 0; k < npairs; ++k) {
            const int s = k % S, m = k % kMmaMStages;
            // the stage's harmonics have landed and the MMAs that read this
            // Mbig stage last (pair k - kMmaMStages) have completed
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)(k / S) & 1u, prm.wait_ns) &&
                                             mbar_wait(&mfree[m], ((uint32_t)(k / kMmaMStages) & 1u) ^ 1u,
                                                       prm.wait_ns))) {
                failed = true;
                break;
            }
            // both slots every time (a slot without an edge computes from stale
            // harmonics into a stage no MMA reads)
            const unsigned char *sha = smem + prm.sh_off + (2 * s) * SHB, *shb = sha + SHB;
            unsigned char *ma = smem + prm.m_off + (4 * m) * MB, *mb = ma + 2 * MB;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const float va = fmaf(e_c0[q], *reinterpret_cast<const float *>(sha + e_j0[q]),
                                      e_c1[q] * *reinterpret_cast<const float *>(sha + e_j1[q]));
                const float vb = fmaf(e_c0[q], *reinterpret_cast<const float *>(shb + e_j0[q]),
                                      e_c1[q] * *reinterpret_cast<const float *>(shb + e_j1[q]));
                const __nv_bfloat16 ha = __float2bfloat16_rn(va), hb = __float2bfloat16_rn(vb);
                *reinterpret_cast<__nv_bfloat16 *>(ma + e_off[q]) = ha;
                *reinterpret_cast<__nv_bfloat16 *>(ma + MB + e_off[q]) = __float2bfloat16_rn(va - __bfloat162float(ha));
                *reinterpret_cast<__nv_bfloat16 *>(mb + e_off[q]) = hb;
                *reinterpret_cast<__nv_bfloat16 *>(mb + MB + e_off[q]) = __float2bfloat16_rn(vb - __bfloat162float(hb));
            }
            fence_proxy_async_smem();  // Mbig is read by the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(&mready[m]);
        }
        if (failed && lane == 0) set_status(prm.status, TP_DEV_ERR_TIMEOUT);
    } else {
        // ================================ MMA issue ================================
        const uint32_t sbase = smem_u32(smem);
        int k_committed = 0;
        if (lane == 0) {
            for (int k = 0; k < npairs; ++k) {
                const int s = k % S, b = k & 1, m = k % kMmaMStages;
                if (!mbar_wait(&mready[m], (uint32_t)(k / kMmaMStages) & 1u, prm.wait_ns) ||
                    !mbar_wait(&tempty[b], ((uint32_t)(k >> 1) & 1u) ^ 1u, prm.wait_ns)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const bool liveA = k < nA, liveB = k < nB;
                const uint32_t d = tmem + (uint32_t)(b * 128);
                const uint32_t xa = sbase + prm.x_off + s * 4096, xb = xa + 2048;
                const uint32_t z0 = sbase + prm.z0_off, z1 = sbase + prm.z1_off;
                const uint32_t m0 = sbase + prm.m_off + (4 * m) * MB;
                // A = [x_A ; 0]: MN atom 0 at x_A, atom 1 at the zero atom after the stages
                const uint64_t a1 = smem_desc(xa, z1 - xa, 1024, 2);
                // A = [0 ; x_B]: MN atom 0 at the zero atom before the stages, atom 1 at x_B
                const uint64_t a2 = smem_desc(z0, xb - z0, 1024, 2);
                if (liveA) {
                    tc_mma_bf16(d, a1, smem_desc(m0, 128, 256, 0), IDESC, false);
                    tc_mma_bf16(d, a1, smem_desc(m0 + MB, 128, 256, 0), IDESC, true);
                }
                if (liveB) {
                    tc_mma_bf16(d, a2, smem_desc(m0 + 2 * MB, 128, 256, 0), IDESC, liveA);
                    tc_mma_bf16(d, a2, smem_desc(m0 + 3 * MB, 128, 256, 0), IDESC, true);
                }
                tc_commit(&mdone[b]);
                tc_commit(&mfree[m]);
                k_committed = k + 1;
            }
            if (failed) {
                set_status(prm.status, TP_DEV_ERR_TIMEOUT);
                // the last committed MMAs finish before tensor memory is released
                for (int k = max(0, k_committed - 2); k < k_committed; ++k)
                    (void)mbar_wait(&mdone[k & 1], (uint32_t)(k >> 1) & 1u, kWaitNs);
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaIssuerWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kMmaTmemCols);
    }
}

}  // namespace tpc
