/*
 * tpconv.h - C ABI of the GB300 (sm_103a) fused equivariant tensor-product
 * convolution library (libtpconv.so).
 *
 * What the library computes. For every edge e of a graph, gather the source
 * node's irreps features x[src[e]], contract them with the edge's real
 * spherical harmonics sh[e] through the real Clebsch-Gordan tensor C_p of
 * every allowed path p = (l_a, l_b, l_c) in channelwise "uvu" mode, scale by
 * the per-edge, per-path, per-channel weight w[e, p, u], and sum into the
 * destination node:
 *
 *   out[d, c, k, u] = sum_{e: dst[e]=d} sum_{p=(a,b,c)} w[e,p,u]
 *                     * sum_{i,j} C_p[i,j,k] x[src[e], a, i, u] sh[e, b, j]
 *
 * This is the descriptor "[ijk]·a[uv]·b[iu]·c[jv] -> D[kuv]" (v = 1) of
 * Lesson 12a: Foundations of cuEquivariance, section 21.4, with the gather
 * (input indices) and sum-scatter (output indices: repeated receivers sum,
 * destinations without edges stay zero) of "cuEquivariance in PyTorch",
 * SegmentedPolynomial: gather and scatter, and external per-edge weights
 * (same page, Layouts and weights: a gathered graph op uses the edge count as
 * the weight batch). All paths run in one kernel with no per-path
 * intermediates (Lesson 12a, section 21.1).
 *
 * Conventions shared by every entry point:
 *  - Feature rows use the ir_mul layout (Lesson 12a, section 21.3): block b of
 *    multiplicity m and degree l occupies (2l+1)*m consecutive elements and
 *    element (i, u) sits at off_b + i*m + u. Blocks follow the irreps string.
 *  - Real basis: m = -l..l with the z axis as pole, l=1 ordered (y, z, x);
 *    spherical harmonics with "component" normalisation (sum_m Y_lm^2 = 2l+1
 *    on unit vectors). Clebsch-Gordan tensors are orthonormal over (i, j) for
 *    each k, with the first nonzero entry in (i, j, k) row-major order
 *    positive. No other normalisation factor is applied.
 *  - Paths: for a in input blocks, b in harmonic blocks, l_o from |l_a-l_b| to
 *    l_a+l_b ascending, kept when (l_o, p_a*p_b) is one of the output types
 *    (Lesson 12a, section 21.4). Paths reaching the same output type sum into
 *    that one output block. Weights are w[e, p*mul + u], path-major.
 *  - Pointers named "device" must be device memory of the current CUDA device;
 *    the caller allocates and owns every buffer. The library owns only the
 *    opaque descriptor (host memory). Every GPU entry point is asynchronous on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and returns a
 *    host-side status for argument errors and launch failures. Problems found
 *    on the device (index out of range, a pipeline wait that gave up) set bits
 *    of a per-device status word read with tp_device_status(); kernels never
 *    trap.
 *  - Indices are int32. Edge counts must be < 2^31.
 */
#ifndef TPCONV_H
#define TPCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TPCONV_ABI_VERSION 1

#if defined(__GNUC__)
#define TPCONV_API __attribute__((visibility("default")))
#else
#define TPCONV_API
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_PARSE = 1,       /* an irreps string cannot be parsed */
    TP_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle (see tp_desc_create) */
    /* 3 is unused: row pointers live in device memory and are checked by the
       kernels, which report bad ones through TP_DEV_ERR_SEGMENT */
    TP_ERR_INDEX = 4,       /* an index is out of range */
    TP_ERR_ALIGN = 5,       /* a pointer or row size breaks the 16-byte rule */
    TP_ERR_CUDA = 6,        /* a CUDA runtime call failed */
    TP_ERR_ARG = 7,         /* null pointer, negative size or bad enum */
    TP_ERR_TIMEOUT = 8,     /* a device pipeline wait gave up (device status bit) */
    TP_ERR_CAPACITY = 9     /* size exceeds a fixed capacity (tp_csr_build_noalloc) */
} tp_status;

typedef enum { TP_IR_MUL = 0, TP_MUL_IR = 1 } tp_layout;

typedef enum {
    TP_F32 = 0,           /* x, w float32; math and out float32 */
    TP_BF16_IN_F32_OUT = 1 /* x, w bfloat16; math (fp32 accumulation) and out float32 */
} tp_dtype;

/* device status bits (tp_device_status) */
#define TP_DEV_ERR_INDEX 0x1   /* src/dst/key outside [0, N) - the edge was skipped */
#define TP_DEV_ERR_TIMEOUT 0x2 /* a pipeline (mbarrier) wait exceeded its time limit; outputs unspecified */
#define TP_DEV_ERR_SEGMENT 0x4 /* row pointers not non-decreasing or outside [0, E] */
#define TP_DEV_ERR_INTERNAL 0x8 /* a kernel's own consistency check failed (a library bug); the access was skipped */

typedef struct tp_desc tp_desc;

typedef struct {
    int32_t n_paths;       /* P */
    int32_t mul;           /* channel multiplicity u (uniform) */
    int32_t dim_x;         /* sum over input blocks of mul*(2l+1) */
    int32_t dim_sh;        /* sum over harmonic blocks of (2l+1) */
    int32_t dim_out;       /* sum over output blocks of mul*(2l+1) */
    int32_t weight_numel;  /* P*mul */
    int32_t n_in, n_sh, n_out; /* number of blocks */
    int32_t lmax_in, lmax_sh, lmax_out;
    int32_t cg_nnz;        /* nonzero Clebsch-Gordan entries over all paths */
    int32_t layout;        /* tp_layout of x and out rows */
} tp_desc_info;

typedef struct {
    int32_t a, b, c;    /* block indices into irreps_in, irreps_sh, irreps_out */
    int32_t la, lb, lc; /* their degrees */
} tp_path_info;

/* Build a descriptor from three irreps strings ("128x0e+128x1o+128x2e",
 * "0e+1o+2e+3o", ...; O(3) with e/o parity letters or SO(3) without,
 * Lesson 12a, section 21.2). The host derives the path table, the real
 * Clebsch-Gordan tensors (Racah's formula in the complex basis, then the
 * complex-to-real change of basis) and the kernel tables.
 * `layout` is the layout of the x and out rows the caller passes (Lesson 12a,
 * section 21.3): TP_IR_MUL, which every entry point takes, or TP_MUL_IR,
 * which tp_conv_forward_ex converts blockwise on the device (the kernels
 * compute in ir_mul); the other entry points return TP_ERR_UNSUPPORTED for a
 * TP_MUL_IR descriptor.
 * Errors: TP_ERR_PARSE for a malformed string; TP_ERR_UNSUPPORTED when
 * a degree exceeds 3, a harmonic block has mul != 1,
 * input/output multiplicities differ or are not one value, an output type
 * repeats, two input (or output) blocks share a degree, mul is not a
 * multiple of 8 or exceeds 128, or no path exists; TP_ERR_ARG for nulls.
 * On success *out owns host memory until tp_desc_destroy. */
TPCONV_API tp_status tp_desc_create(const char *irreps_in, const char *irreps_sh, const char *irreps_out,
                         tp_layout layout, tp_desc **out);
/* A descriptor whose output has one block per path ("unsimplified", as the
 * descriptor printout of Lesson 12a, section 21.4: 32x0e+32x1o x 0e+1o gives
 * D=32x0e+32x0e+32x1o+32x1o) instead of one per output type: irreps_out
 * lists the allowed output types; path p writes its own block of
 * mul*(2l_c+1) elements; blocks are grouped by output type in the order of
 * irreps_out, paths of one type in path order. tp_desc_query reports that
 * output width and n_out = n_paths; tp_desc_path reports a path's block as c.
 * tp_conv_forward (and tp_conv_forward_ex with reduce sum, int32 or int64
 * indices) accept it; layout must be TP_IR_MUL, and every other entry point
 * returns TP_ERR_UNSUPPORTED for it. */
TPCONV_API tp_status tp_desc_create_unsimplified(const char *irreps_in, const char *irreps_sh,
                                                 const char *irreps_out, tp_layout layout, tp_desc **out);
TPCONV_API tp_status tp_desc_query(const tp_desc *desc, tp_desc_info *info);
/* Path p in enumeration order (the weight layout order). */
TPCONV_API tp_status tp_desc_path(const tp_desc *desc, int32_t p, tp_path_info *info);
/* Copy path p's dense Clebsch-Gordan tensor [2la+1][2lb+1][2lc+1] (row-major,
 * float64) into host memory `out` of `capacity` doubles. */
TPCONV_API tp_status tp_desc_cg(const tp_desc *desc, int32_t p, double *out, int64_t capacity);
TPCONV_API void tp_desc_destroy(tp_desc *desc);

/* Real spherical harmonics of the desc's harmonic irreps for E edge vectors
 * ("cuEquivariance in PyTorch", Spherical harmonics and a NumPy reference:
 * normalize != 0 first scales each vector to unit length; normalize == 0
 * evaluates the raw homogeneous polynomial).
 * vec: device float32 [E][3]; sh: device float32 [E][dim_sh]. */
TPCONV_API tp_status tp_spherical_harmonics(const tp_desc *desc, const float *vec, int64_t E, int32_t normalize,
                                 float *sh, void *stream);

/* Workspace bytes tp_csr_build needs for E keys in [0, N). */
TPCONV_API tp_status tp_csr_workspace_size(int64_t E, int32_t N, size_t *bytes);

/* Stable counting sort of keys (a dst-sorted CSR when keys = dst; a source
 * CSR for the backward when keys = src in dst-sorted edge order). The
 * destination-sorted edge list is what the gather/scatter of "cuEquivariance
 * in PyTorch", SegmentedPolynomial: gather and scatter, sums over (one
 * contiguous edge range per output row), and the same page's Limitations and
 * backends notes that indexed kernels want sorted indices.
 * keys: device int32 [E] in [0, N). Outputs (device, caller-owned):
 *   perm[E]         perm[k] = original position of the k-th sorted key; equal
 *                   keys keep their original order;
 *   row_ptr[N+1]    row_ptr[0] = 0, row_ptr[N] = E, segment d = [row_ptr[d], row_ptr[d+1]);
 *   keys_sorted[E]  optional (NULL to skip).
 * workspace: device memory of at least tp_csr_workspace_size bytes, 256-byte
 * aligned. Keys outside [0, N) set TP_DEV_ERR_INDEX; outputs are then
 * unspecified but every write stays inside the output arrays. */
TPCONV_API tp_status tp_csr_build(const int32_t *keys, int64_t E, int32_t N, int32_t *perm, int32_t *row_ptr,
                       int32_t *keys_sorted, void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free tp_csr_build. The pages have no counterpart: this entry
 * point is for callers that cannot allocate device memory themselves, such as
 * a plugin whose enqueue callback of a host framework receives only the
 * tensors it reads and writes, or a program whose device memory is entirely
 * owned by another allocator, where an extra cudaMalloc would fail, break the
 * allocator's accounting, or synchronise the device. Results are identical to
 * tp_csr_build.
 * The sort's scratch is a fixed array inside the library (about 3.3 MB, held on
 * every GPU that loads the library until the process exits); the caller still
 * passes keys and the outputs. E may be at most
 * tp_csr_build_noalloc_max_edges() (262144); larger E returns TP_ERR_CAPACITY
 * without launching anything. The first call on each device looks up the
 * array's device address with a runtime query (a one-time set-up, no
 * allocation). All calls share the one array, so
 * calls that overlap on the GPU (different streams, or different host
 * threads) race and must be serialised by the caller. Nothing in the array
 * needs to start at zero: every call overwrites what it reads. */
TPCONV_API tp_status tp_csr_build_noalloc(const int32_t *keys, int64_t E, int32_t N, int32_t *perm,
                                          int32_t *row_ptr, int32_t *keys_sorted, void *stream);
TPCONV_API int64_t tp_csr_build_noalloc_max_edges(void);

/* Forward pass (the hot path): the formula at the top of this file, that is
 * the channelwise product "[ijk]·a[uv]·b[iu]·c[jv] -> D[kuv]" of Lesson 12a:
 * Foundations of cuEquivariance, section 21.4, with x gathered by source and
 * the result sum-scattered by destination ("cuEquivariance in PyTorch",
 * SegmentedPolynomial: gather and scatter; one weight row per edge as in
 * Layouts and weights), every path in one launch (Lesson 12a, section 21.1).
 * Edges must be in destination-sorted order with row_ptr[N_dst+1] from
 * tp_csr_build (edge range of destination d is [row_ptr[d], row_ptr[d+1])).
 *   x:   device [N_src][dim_x], float32 (TP_F32) or bfloat16 (TP_BF16_IN_F32_OUT), ir_mul;
 *   sh:  device float32 [E][dim_sh];
 *   w:   device [E][weight_numel], same type as x;
 *   src: device int32 [E], in [0, N_src);
 *   out: device float32 [N_dst][dim_out], fully overwritten (zero rows for
 *        destinations without edges);
 *   workspace: device memory of tp_conv_forward_workspace_size() bytes
 *        (256-byte aligned), or NULL. It holds the partial rows of destinations
 *        that straddle the kernel's exact, edge-balanced split of the edge list
 *        into pieces (0 bytes are reported when the descriptor has no split
 *        kernel). A smaller workspace makes the split use fewer pieces; with
 *        NULL, or when sh is not 16-byte aligned, the library uses its generic
 *        kernel, which needs none but splits work per destination.
 * x, w and out must be 16-byte aligned; dim_x*sizeof(x) and
 * weight_numel*sizeof(w) must be multiples of 16 (they are whenever mul % 8
 * == 0). An out-of-range src entry sets TP_DEV_ERR_INDEX and its edge adds
 * nothing. Summation order is fixed: results are bitwise reproducible run to
 * run on one device (the split depends on the device's SM count and on the
 * workspace size). */
TPCONV_API tp_status tp_conv_forward_workspace_size(const tp_desc *desc, tp_dtype dtype, int32_t N_dst, int64_t E,
                                                    size_t *bytes);
TPCONV_API tp_status tp_conv_forward(const tp_desc *desc, tp_dtype dtype, const void *x, const float *sh,
                                     const void *w, const int32_t *src, const int32_t *row_ptr, int32_t N_src,
                                     int32_t N_dst, int64_t E, float *out, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* tp_conv_forward with the spherical harmonics evaluated inside the kernel
 * from edge vectors, so the per-edge harmonic rows never pass through device
 * memory ("cuEquivariance in PyTorch", Trainable message passing: the
 * convolution is fed sh(edge_vectors); Spherical harmonics and a NumPy
 * reference: normalize != 0 takes the harmonics of the unit vector, a zero
 * vector then giving Y_0 = 1 and zeros; normalize == 0 the raw homogeneous
 * polynomial). vec: device float32 [E][3] in the destination-sorted edge order,
 * 16-byte aligned; every other argument as for tp_conv_forward. The harmonics
 * are those of the descriptor's harmonic irreps, which must be blocks 0..L in
 * order (the layout the compiled kernels use). Needs a workspace of
 * tp_conv_forward_workspace_size() bytes; TP_ERR_UNSUPPORTED when the
 * descriptor has no compiled kernel, the workspace is missing or too small. */
TPCONV_API tp_status tp_conv_forward_vec(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const void *w, const int32_t *src,
                                         const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                                         float *out, void *workspace, size_t workspace_bytes, void *stream);

/* Radial network producing the per-edge weights from the edge length
 * ("cuEquivariance in PyTorch", Trainable message passing: weights =
 * radial(|edge_vector|) with radial = Linear(1, 16) -> SiLU -> Linear(16,
 * weight_numel)):
 *   h[i] = silu(w1[i] * |v| + b1[i]),  silu(z) = z / (1 + exp(-z)),  i < hidden
 *   w[j] = b2[j] + sum_i w2[i * weight_numel + j] * h[i],             j < weight_numel
 * All pointers are device float32: w1[hidden], b1[hidden], w2[hidden][weight_numel]
 * (hidden-major, i.e. the transpose of a torch Linear(hidden, weight_numel)
 * weight), b2[weight_numel]. hidden must be 16. w1 and b1 4-byte aligned, w2
 * and b2 16-byte aligned (the kernels read w2 and b2 in 16-byte pieces);
 * TP_ERR_ALIGN otherwise. */
typedef struct {
    const float *w1, *b1;
    const float *w2, *b2;
    int32_t hidden;
} tp_radial_mlp;

/* tp_conv_forward_vec with the per-edge weights computed inside the kernel by
 * the radial network from the edge length, so the weight stream (the dominant
 * bytes of the plain forward) is never read from or written to device memory.
 * float32 only (dtype must be TP_F32); every other argument as for
 * tp_conv_forward_vec. TP_ERR_UNSUPPORTED for other dtypes, mlp->hidden != 16,
 * or a descriptor without a compiled kernel / too small a workspace. */
TPCONV_API tp_status tp_conv_forward_mlp(const tp_desc *desc, tp_dtype dtype, const void *x, const float *vec,
                                         int32_t normalize, const tp_radial_mlp *mlp, const int32_t *src,
                                         const int32_t *row_ptr, int32_t N_src, int32_t N_dst, int64_t E,
                                         float *out, void *workspace, size_t workspace_bytes, void *stream);

/* Reductions over a destination's incoming edges ("cuEquivariance in PyTorch",
 * Other operations and layers: the convolution layer supports reduce="mean").
 * SUM: the formula at the top of this file; MEAN: that sum divided by the
 * destination's number of edges (destinations without edges stay zero). */
#define TP_REDUCE_SUM 0
#define TP_REDUCE_MEAN 1

/* Arguments of tp_conv_forward_ex. The harmonics come either as rows `sh`
 * [E][dim_sh] or, with `vec` [E][3] non-NULL instead, are evaluated in the
 * kernel (as tp_conv_forward_vec; `normalize` as there); with `mlp` (needs
 * `vec`) the weights come from the radial network (as tp_conv_forward_mlp) and
 * `w` is ignored. x and out rows are in the descriptor's layout; src
 * [E] and row_ptr [N_dst+1] are int32 (index_bits 32) or int64 (index_bits 64,
 * "cuEquivariance in PyTorch", SegmentedPolynomial: gather and scatter: index
 * tensors may be int32 or int64; values must fit int32). The workspace (256-byte
 * aligned, tp_conv_forward_ex_workspace_size bytes) is required. */
typedef struct {
    tp_dtype dtype;
    const void *x;
    const float *sh;
    const float *vec;
    int32_t normalize;
    const tp_radial_mlp *mlp;
    const void *w;
    const void *src;
    const void *row_ptr;
    int32_t index_bits;
    int32_t reduce;
    int32_t N_src, N_dst;
    int64_t E;
    float *out;
    void *workspace;
    size_t workspace_bytes;
} tp_forward_args;

/* The forward with int64 indices, a TP_MUL_IR descriptor or TP_REDUCE_MEAN.
 * Around the same fused kernels it runs, on `stream`: int64 -> int32 copies of
 * src and row_ptr (an index outside int32 becomes -1, which the kernels flag
 * and skip); a blockwise mul_ir -> ir_mul copy of x and an ir_mul -> mul_ir copy
 * of out; the mean scaling of each row. Errors as tp_conv_forward, plus
 * TP_ERR_ARG for a missing or small workspace, both sh and vec, or a bad
 * index_bits / reduce. */
TPCONV_API tp_status tp_conv_forward_ex_workspace_size(const tp_desc *desc, const tp_forward_args *args,
                                                       size_t *bytes);
TPCONV_API tp_status tp_conv_forward_ex(const tp_desc *desc, const tp_forward_args *args, void *stream);

/* Blockwise layout conversion of `rows` feature rows of the descriptor's input
 * (which = 0) or output (which = 1) irreps between mul_ir and ir_mul (Lesson
 * 12a, section 21.3; "cuEquivariance in PyTorch", Layouts and weights: the
 * conversion is per irrep block, not of the whole flattened row). `from` is the
 * layout of src; dst receives the other one. src and dst: device, elem_bytes
 * 2 or 4 per element, distinct, [rows][dim]. */
TPCONV_API tp_status tp_transpose_layout(const tp_desc *desc, int32_t which, tp_layout from, const void *src,
                                         void *dst, int64_t rows, int32_t elem_bytes, void *stream);

/* Backward pass of tp_conv_forward, the exact gradients of <grad_out, out>
 * with respect to x, w and sh ("cuEquivariance in PyTorch", CPU tensor
 * product and backward: gradients with respect to both inputs and the
 * weights; the forward is linear in each of them, so these sums are exact):
 *   dx[s,a,i,u] = sum_{e: src[e]=s} sum_{p: a_p=a} w[e,p,u] sum_{j,k} C_p[i,j,k] sh[e,b,j] g[dst[e],c,k,u]
 *   dw[e,p,u]   = sum_{i,j,k} C_p[i,j,k] x[src[e],a,i,u] sh[e,b,j] g[dst[e],c,k,u]
 *   dsh[e,b,j]  = sum_{p: b_p=b} sum_{i,k,u} C_p[i,j,k] x[src[e],a,i,u] w[e,p,u] g[dst[e],c,k,u]
 * dtype TP_F32: x and w float32; TP_BF16_IN_F32_OUT: x and w bfloat16 (the
 * forward's bfloat16 inputs), every product and sum in float32. grad_out
 * [N_dst][dim_out], sh [E][dim_sh] and all three gradients are float32.
 * Edges are in destination-sorted order (row_ptr as for the forward; dst[E]
 * the sorted destination of each edge). The source CSR (src_perm, src_row_ptr)
 * is tp_csr_build of `src` in that same edge order: src_perm lists edge
 * positions grouped by source. dx [N_src][dim_x], dw [E][weight_numel] and
 * dsh [E][dim_sh] are fully overwritten (for every edge src_perm lists; an
 * edge whose destination is out of range gets zero dw and dsh rows and sets
 * TP_DEV_ERR_INDEX). Deterministic (no atomics).
 * workspace: device memory of tp_conv_backward_workspace_size bytes (16-byte
 * aligned) for the partial dx rows of sources whose edges two warps share;
 * with a smaller (or NULL) workspace the call uses fewer warps, or the
 * generic two-kernel backward (float32 only). TP_ERR_UNSUPPORTED for
 * bfloat16 inputs when the descriptor has no compiled path program. */
TPCONV_API tp_status tp_conv_backward_workspace_size(const tp_desc *desc, tp_dtype dtype, int32_t N_src, int64_t E,
                                                     size_t *bytes);
TPCONV_API tp_status tp_conv_backward(const tp_desc *desc, tp_dtype dtype, const float *grad_out, const void *x,
                                      const float *sh, const void *w, const int32_t *src, const int32_t *dst,
                                      const int32_t *row_ptr, const int32_t *src_perm, const int32_t *src_row_ptr,
                                      int32_t N_src, int32_t N_dst, int64_t E, float *dx, float *dw, float *dsh,
                                      void *workspace, size_t workspace_bytes, void *stream);

/* Launch tuning and test hooks. The pages have no counterpart: these settings
 * exist for tests and tuning sweeps, and normal use never needs them. They
 * are process-wide and apply to calls made after tp_set_tuning returns; a zero
 * field keeps the library's default.
 *   ring_stage_bytes  target bytes per chunk of the forward's warp ring (>= 0)
 *   ring_stages       stages per warp ring, 2..8
 *   ring_warps        warps per block of the ring kernel, 1..8
 *   ring_rounds       pieces of the edge list per warp, 1..16
 *   ring_pack         1: packed two-lane FMAs, 2: plain FMAs
 *   disable_split     1: the forward uses its generic per-destination kernel
 *   wait_limit_ns     time after which a kernel's main-loop pipeline wait gives
 *                     up and sets TP_DEV_ERR_TIMEOUT (default 1 s); waits that
 *                     let a failed warp's copies land before it exits always
 *                     keep the 1 s limit.
 *   disable_mma       1: bfloat16 inputs skip the tensor-core kernel
 *   mma_stages        shared-memory stages of the tensor-core kernel, 3..8
 *   bwd_stage_bytes   target bytes per chunk of the backward's warp ring (>= 0)
 *   bwd_stages        stages per backward warp ring, 2..8
 *   bwd_warps         warps per block of the backward ring kernel, 1..8
 *   disable_ring_bwd  1: float32 backward uses the generic two-kernel path
 *   disable_symc_jit  1: the symmetric contraction uses its table kernel
 *                     instead of the kernel compiled for the descriptor
 * tp_set_tuning(NULL) restores every default. TP_ERR_ARG for a field out of range. */
typedef struct {
    int32_t ring_stage_bytes;
    int32_t ring_stages;
    int32_t ring_warps;
    int32_t ring_rounds;
    int32_t ring_pack;
    int32_t disable_split;
    int64_t wait_limit_ns;
    int32_t disable_mma;
    int32_t mma_stages;
    int32_t bwd_stage_bytes;
    int32_t bwd_stages;
    int32_t bwd_warps;
    int32_t disable_ring_bwd;
    int32_t disable_symc_jit;
} tp_tuning;
TPCONV_API tp_status tp_set_tuning(const tp_tuning *tuning);
TPCONV_API tp_status tp_get_tuning(tp_tuning *tuning);

/* Symmetric contraction (MACE-style; Lesson 12a, section 21.4.1: one line per
 * body order nu, "[]·a[u]·b[u]·...·b[u] -> C[u]"; "cuEquivariance in PyTorch",
 * Other operations and layers: uniform multiplicities, a contraction degree,
 * a number of elements and integer element indices). Per node n and channel u,
 * with b[n, i, u] the components of every input block of the node's features:
 *   out[n, c, k, u] = sum_{nu=1..max_degree} sum_q a[element[n], q, u]
 *                     * sum_{i_1..i_nu} B_q[i_1..i_nu, k] prod_t b[n, i_t, u]
 * The basis tensors B_q of each (nu, output block) span the tensors symmetric
 * in the nu slots and equivariant under rotations (and inversions for O(3));
 * they are made canonical by the reduced row echelon form of the spanning set
 * (flattened row-major over (i_1..i_nu, k)), each scaled to unit norm with a
 * positive leading entry. For 32x0e+32x1o -> 32x0e and degrees 1..3 that is
 * 1, 2 and 2 weights per channel with 1, 4 and 10 nonzero entries, as printed
 * on the lesson. Weights are ordered term by term: degree ascending, then
 * output block, then basis tensor. */
typedef struct tp_symc tp_symc;
typedef struct {
    int32_t mul, dim_in, dim_out, max_degree;
    int32_t n_weights;             /* per element and channel */
    int32_t n_terms;               /* (degree, output block) pairs with a basis */
    int32_t num_paths[3];          /* nonzero basis entries of degree 1, 2, 3 */
    int32_t weights_per_degree[3];
} tp_symc_info;
/* irreps_in: input blocks of degrees <= 2, one multiplicity (a multiple of 32);
 * irreps_out: output blocks of degrees <= 3, the same multiplicity; max_degree
 * 1..3. TP_ERR_PARSE / TP_ERR_UNSUPPORTED / TP_ERR_ARG as tp_desc_create. */
TPCONV_API tp_status tp_symc_create(const char *irreps_in, const char *irreps_out, int32_t max_degree,
                                    tp_symc **out);
TPCONV_API tp_status tp_symc_query(const tp_symc *symc, tp_symc_info *info);
/* Term t: its degree, output block, number of basis tensors and (when basis
 * is not NULL) the dense basis [n_q][D]..[D][2L+1] as float64 into host memory
 * of `capacity` doubles. */
TPCONV_API tp_status tp_symc_term(const tp_symc *symc, int32_t t, int32_t *nu, int32_t *out_block, int32_t *n_q,
                                  double *basis, int64_t capacity);
TPCONV_API void tp_symc_destroy(tp_symc *symc);
/* The CUDA source of the kernel tp_symmetric_contraction compiles for this
 * descriptor (at run time, with NVRTC, once per device): the basis as
 * straight-line code. Writes up to `capacity` bytes (NUL-terminated when it
 * fits) into host memory `buf` and the full length (without the NUL) into
 * *length. For inspection and tests; needs no GPU. */
TPCONV_API tp_status tp_symc_kernel_source(const tp_symc *symc, char *buf, int64_t capacity, int64_t *length);
/* x: device float32 [N][dim_in] (ir_mul), 16-byte aligned; weights: device
 * float32 [num_elements][n_weights][mul], 8-byte aligned; element: device
 * int32 [N] in [0, num_elements) (an index outside sets TP_DEV_ERR_INDEX and
 * the node's row is zero); out: device float32 [N][dim_out] (ir_mul), 16-byte
 * aligned, fully overwritten. Misaligned pointers give TP_ERR_ALIGN; a basis
 * with more than 2000 nonzero entries or 512 (output row, weight) pairs gives
 * TP_ERR_UNSUPPORTED. Asynchronous on `stream`; nothing is allocated. */
TPCONV_API tp_status tp_symmetric_contraction(const tp_symc *symc, const float *x, const float *weights,
                                              const int32_t *element, int32_t N, int32_t num_elements, float *out,
                                              void *stream);

/* Read (and, when reset != 0, clear) the current device's status word into
 * *flags (TP_DEV_ERR_* bits). Synchronises `stream`. */
TPCONV_API tp_status tp_device_status(int32_t *flags, int32_t reset, void *stream);

TPCONV_API const char *tp_status_string(tp_status status);
TPCONV_API int32_t tp_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TPCONV_H */
