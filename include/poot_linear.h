/*
 * poot_linear.h -- C ABI of the GB300 (sm_103a) FP16 linear library.
 *
 * One operation:  y = FP16(x . W^T) + b
 *
 *   x  [M, K]  row-major binary16, one input row per output row
 *   W  [N, K]  row-major binary16, [out_features, in_features]; the kernels
 *              read it in this layout (the transpose is never formed)
 *   b  [N]     binary16, the same b[n] for every row
 *   y  [M, N]  row-major binary16
 *
 * Numerical contract ("Tensor Programs, Part 1", section "One Program and One
 * Numerical Contract", the proj formula and rules 1-2, and the Figure 1.1
 * caption):
 *   1. the products x[m,k] * W[n,k] enter an FP32 sum unrounded (each product
 *      of two binary16 numbers is exact in binary32); the summation order is
 *      free;
 *   2. proj[m,n] = RN16(sum) is rounded to binary16 BEFORE the bias, then
 *      y[m,n] = RN16(proj[m,n] + b[n]).  proj lives only in registers.
 * RN16 is IEEE round-to-nearest-even with gradual underflow and overflow to
 * infinity.
 *
 * All entry points are plain C: device pointers and sizes, no torch types.
 * All functions return a status code (POOT_OK or a POOT_ERR_* value) and
 * never abort the process; an error is reported, not raised.
 */
#ifndef POOT_LINEAR_H
#define POOT_LINEAR_H

#include <stdint.h>

#if defined(__GNUC__)
#define POOT_API __attribute__((visibility("default")))
#else
#define POOT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t); NULL is the legacy default
 * stream of the calling thread's current device. */
typedef struct CUstream_st* poot_stream_t;

/* ---- status codes ------------------------------------------------------- */
enum {
    POOT_OK = 0,
    POOT_ERR_INVALID_ARG = 1,        /* NULL pointer, negative or too large
                                        dimension, y overlapping an input,
                                        an unknown or inapplicable variant */
    POOT_ERR_MISALIGNED = 2,         /* a pointer is not 2-byte aligned */
    POOT_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 */
    POOT_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed;
                                        poot_linear_last_cuda_error() names it */
    POOT_ERR_DEVICE_TIMEOUT = 5      /* a kernel's bounded wait ran out */
};

/* ---- kernel variants (the plan-time GEMV / GEMM split) ------------------ */
enum {
    POOT_VARIANT_AUTO = -1,       /* choose from M, N, K and pointer alignment */
    POOT_VARIANT_NONE = 0,        /* M == 0 or N == 0: nothing to do */
    POOT_VARIANT_BIAS_ONLY = 1,   /* K == 0: y[m,n] = RN16(+0 + b[n]) */
    POOT_VARIANT_GEMV = 2,        /* M <= 16: HBM-bound weight stream,
                                     128-bit loads (K % 8 == 0, x and W
                                     16-byte aligned) */
    POOT_VARIANT_GEMV_SCALAR = 3, /* M <= 16, any K and alignment */
    POOT_VARIANT_GEMM_TMA = 4,    /* tcgen05 GEMM, TMA loads of x and W
                                     (K % 8 == 0, x and W 16-byte aligned) */
    POOT_VARIANT_GEMM_CPASYNC = 5,/* tcgen05 GEMM, 4-byte async copies for
                                     row pitches TMA cannot take
                                     (K even, x and W 4-byte aligned) */
    POOT_VARIANT_GEMM_REG = 6,    /* tcgen05 GEMM, 2-byte register copies
                                     (any K and alignment) */
    POOT_VARIANT_GEMM_PACKED = 7  /* any K and alignment: a copy kernel
                                     writes x and W with rows padded to a
                                     16-byte pitch into the library's
                                     workspace ((M + N) * ceil8(K) * 2
                                     bytes, as for split-K), then the TMA
                                     GEMM runs on the copies.  The choice
                                     for M > 16 when TMA cannot read x or W
                                     in place; if no workspace can be had it
                                     runs as GEMM_CPASYNC or GEMM_REG */
};

/* Largest M served by the GEMV variants. */
#define POOT_GEMV_MAX_M 16

/*
 * y = FP16(x . W^T) + b on the calling thread's current device.
 *
 * Source: "Tensor Programs, Part 1", the toy linear y = matmul(x, weight.T) + b
 * and its numerical contract (section "One Program and One Numerical
 * Contract"); the call mirrors the linear(builder, h, weight, bias) op of
 * the poot "Tracing a Model" page.
 *
 * x, w, b, y: device pointers (memory of the current device) to contiguous
 *   row-major binary16 data with the shapes above.  2-byte alignment is
 *   required.  With x and w 16-byte aligned and K % 8 == 0 the GEMM reads
 *   them in place by TMA; otherwise (M > 16) it first copies them into
 *   16-byte-pitched rows (GEMM_PACKED).  y 16-byte aligned with N % 8 == 0
 *   is stored by TMA, else by plain stores.  Every path gives results
 *   within the same contract.
 * M, N, K: sizes, 0 <= M, N, K < 2^31.  M == 0 or N == 0 launches nothing
 *   (pointers may then be NULL).  K == 0 gives y = b in every row (x and w
 *   may then be NULL).
 * stream: the work is queued on it; the call does not synchronise.
 * Ownership: the caller owns all four buffers.  x, w and b are only read;
 *   every element of y is written.  y must not overlap x, w or b.  The
 *   library allocates nothing per call, except that a split-K plan (small
 *   M, long K; see gemm_split_k) and the GEMM_PACKED variant (x or W not
 *   readable by TMA in place) take their workspace from a buffer the
 *   library keeps per device and stream, allocating or growing it on first
 *   need (a graph-owned block under stream capture).
 * Errors: argument errors are found before any CUDA call and nothing is
 *   queued.  Launch failures return POOT_ERR_CUDA.  Faults inside a kernel
 *   surface at the caller's next synchronisation, as for any CUDA kernel;
 *   a bounded device-side wait that runs out is reported by
 *   poot_linear_device_status().
 */
POOT_API int poot_linear_f16(const void* x, const void* w, const void* b, void* y,
                    int64_t M, int64_t N, int64_t K, poot_stream_t stream);

/* Tuning knobs of poot_linear_f16_ex; zero-initialise and set what you need. */
typedef struct poot_linear_options {
    int variant;             /* POOT_VARIANT_AUTO (-1) or a POOT_VARIANT_* code;
                                0 here means POOT_VARIANT_NONE, so set it */
    int gemv_warps_per_row;  /* 0 = automatic; 1, 2, 4 or 8 warps of the GEMV
                                split one output feature's K range.  For
                                3 <= M <= 16 a non-zero value also selects
                                the CUDA-core GEMV instead of the tensor-core
                                one */
    int gemm_tile_n;         /* 0 = automatic; else the GEMM's output tile
                                width: a multiple of 32 in [64, 256] */
    int gemm_group_m;        /* 0 = automatic; else the number of 128-row
                                blocks walked together for L2 reuse (>= 1) */
    int gemm_k_chunk;        /* 0 = automatic (1024; 2048 for contractions
                                with epilogue steps); else a multiple of 64:
                                how many K elements the tensor core sums
                                before the partial sums are added, in IEEE
                                FP32, into the running sum.  A value >= K
                                keeps the whole sum on the tensor core */
    int gemm_cluster;        /* 0 = automatic; 1 = one CTA per 128-row tile;
                                2 = CTA pairs sharing each W tile on 256-row
                                tiles (2-SM MMA); needs the GEMM_TMA or
                                GEMM_PACKED variant.  Any other value is
                                POOT_ERR_INVALID_ARG */
    int gemm_split_k;        /* 0 = automatic; 1 = never; S in [2, 16] = cut
                                the K range into S ranges of whole 64-element
                                blocks (S must divide ceil(K / 64)), each
                                summed by its own tiles into an FP32
                                workspace, then added in range order by a
                                second kernel that applies the epilogue.
                                The workspace (S * M * N * 4 bytes) belongs to
                                the library: one per device and stream, kept
                                for the life of the process; under stream
                                capture, a graph-owned allocation freed on
                                the stream after the second kernel.  Not with
                                grouped contractions.
                                Automatic splitting happens when one wave of
                                output tiles leaves more than a quarter of
                                the SMs idle and K is at least 1024; the tile
                                width and the split are then chosen
                                together.  When no workspace can be had, an
                                automatic split falls back to none and a
                                requested one returns POOT_ERR_CUDA */
} poot_linear_options;

/*
 * Same operation with explicit choices (tests, benchmarks, tuning).
 * opts: may be NULL (everything automatic).  A variant whose preconditions
 *   the arguments do not meet, or an out-of-range knob, returns
 *   POOT_ERR_INVALID_ARG and queues nothing.  The knobs change the work
 *   decomposition only; every choice gives a result within the numerical
 *   contract above.
 */
POOT_API int poot_linear_f16_ex(const void* x, const void* w, const void* b, void* y,
                                int64_t M, int64_t N, int64_t K,
                                const poot_linear_options* opts, poot_stream_t stream);

/*
 * The variant poot_linear_f16 would run for these arguments (pure host
 * logic: pointers are inspected for alignment only, never dereferenced; no
 * CUDA call).  Returns a POOT_VARIANT_* code >= 0, or -POOT_ERR_* when the
 * arguments are invalid.
 */
POOT_API int poot_linear_f16_variant(const void* x, const void* w, const void* b, const void* y,
                            int64_t M, int64_t N, int64_t K);

/*
 * The GEMM's tile plan for y = FP16(x . W^T) + b with x and W readable by
 * TMA in place and every option automatic, on a device with `sm_count` SMs
 * (pure host logic, no CUDA call: tests and benchmarks use it to see which
 * plan runs).  Errors: POOT_ERR_INVALID_ARG for sizes outside [1, 2^31),
 * sm_count < 2 or a NULL out.
 */
typedef struct poot_gemm_plan {
    int tile_n;     /* output tile width (the MMA's N) */
    int cluster;    /* 1: single CTAs, 128-row tiles; 2: CTA pairs, 256-row tiles */
    int split_k;    /* K ranges summed by separate tiles (1: none) */
    int k_chunk;    /* K elements per TMEM accumulation chain */
    int tiles;      /* output tiles (times split_k) */
    int ctas;       /* CTAs of a full grid (persistent: at most one per SM) */
} poot_gemm_plan;
POOT_API int poot_linear_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count, poot_gemm_plan* out);

/* Static, NUL-terminated description of a status code (never NULL). *//* Static, NUL-terminated description of a status code (never NULL). */
POOT_API const char* poot_linear_status_string(int status);

/* Name of the CUDA error behind the calling thread's last POOT_ERR_CUDA
 * (static string; "cudaSuccess" if there was none). */
POOT_API const char* poot_linear_last_cuda_error(void);

/*
 * Synchronises `stream`, then reports and clears the current device's
 * device-side error word: POOT_ERR_DEVICE_TIMEOUT if a kernel's bounded
 * wait ran out since the last call, POOT_ERR_CUDA if the synchronisation
 * failed, else POOT_OK.
 */
POOT_API int poot_linear_device_status(poot_stream_t stream);

/* ---- The widened contraction ---------------------------------------------
 *
 * "ML compiler internals", section "The OpKind vocabulary": the
 * ContractionEpilogue row (a dense contraction and the single-use
 * pointwise chain that consumes it; the head's result keeps its dtype, a
 * BF16 head rounds to BF16 before the first step reads it, and every step
 * rounds through it) and the DenseContraction row (an f32 result); section
 * "SwiGLU and GeLU FFN" (SiLU and GELU are compositions of the Neg, Exp,
 * Add, Div, Mul and Erf primitives).  For every output element
 *
 *   S = sum_k x[m,k] W[n,k]            products in FP32, any summation order
 *   out_f32:  y = S, or RN32(S + b[n]) with a bias   (float32 y, no steps)
 *   else:     t = RN_h(S); t = RN_h(t + b[n]) when b != NULL;
 *             each step:  t = step(t);  y = t         (head dtype h)
 *
 * where every primitive of a step rounds to h:
 *   POOT_EP_ADD        t + r[m,n]
 *   POOT_EP_MUL        t * r[m,n]
 *   POOT_EP_SILU       t / (1 + exp(-t))                 (Neg, Exp, Add, Div)
 *   POOT_EP_GELU_TANH  t / (1 + exp(-c2 (t + c1 t^3))),   c1 = RN_h(0.044715),
 *                      c2 = RN_h(2 sqrt(2/pi))            (Mul, Add, Neg, Exp, Div)
 *   POOT_EP_GELU_ERF   0.5 (t (1 + erf(c3 t))),           c3 = RN_h(1/sqrt 2)
 *                                                          (Mul, Erf, Add)
 * in the order the steps are listed.  Exp and Erf are evaluated in FP32 and
 * rounded to h; every other primitive equals the correctly rounded h result.
 */
enum poot_dtype { POOT_DTYPE_F16 = 0, POOT_DTYPE_BF16 = 1 };
enum poot_epilogue_op {
    POOT_EP_ADD = 1,
    POOT_EP_MUL = 2,
    POOT_EP_SILU = 3,
    POOT_EP_GELU_TANH = 4,
    POOT_EP_GELU_ERF = 5
};
#define POOT_EPILOGUE_MAX_STEPS 4

typedef struct poot_epilogue_step {
    int op;                  /* POOT_EP_* */
    const void* operand;     /* ADD, MUL: device pointer to r, [M, ld] row-major
                                in the head dtype (2-byte aligned, read only,
                                not overlapping y); NULL for the others */
    int64_t ld;              /* row pitch of r in elements (>= N); 0 means N */
} poot_epilogue_step;

typedef struct poot_contraction_spec {
    int dtype;               /* POOT_DTYPE_F16 or POOT_DTYPE_BF16: x, W, b, the
                                step operands and (unless out_f32) y */
    int out_f32;             /* 1: y is float32 (4-byte aligned) and holds the
                                unrounded sum (+ b), num_steps must be 0 */
    int num_steps;           /* 0 .. POOT_EPILOGUE_MAX_STEPS */
    poot_epilogue_step steps[POOT_EPILOGUE_MAX_STEPS];
} poot_contraction_spec;

/*
 * y = the widened contraction of x [M,K] and W [N,K] ([out, in], read in
 * place) with the optional bias b [N] (NULL: none) under `spec`, on
 * `stream`.  All pointers are device pointers; y is [M,N] row-major.
 * M <= 16 (per group) with x and W 16-byte aligned and K % 8 == 0 runs on
 * the GEMV kernels with a per-element epilogue (unless a GEMM split is
 * requested); everything else on the tcgen05 GEMM.  `opts` may be NULL; of
 * its variants POOT_VARIANT_GEMV (where the GEMV applies) and the GEMM ones
 * are accepted, and its GEMV warp split is ignored.  Asynchronous; the caller owns every
 * buffer; the library allocates nothing except the workspace described
 * under poot_linear_f16 (split-K, never for the grouped form; the packed
 * copies of x and W when TMA cannot read them in place).
 * Errors: POOT_ERR_INVALID_ARG for a NULL spec, x, w or y, K == 0, a bad
 * dtype, step code, step count, NULL operand or ld < N, steps with out_f32,
 * or y overlapping x, W, b or an operand; POOT_ERR_MISALIGNED for a pointer
 * below its element alignment; otherwise as poot_linear_f16.
 */
POOT_API int poot_contract(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N,
                           int64_t K, const poot_contraction_spec* spec, const poot_linear_options* opts,
                           poot_stream_t stream);

/*
 * Grouped contraction: G independent contractions in one launch, the
 * GroupedDenseContraction row of the OpKind table ("ML compiler
 * internals", section "The OpKind vocabulary": a [G*N, K] weight read in
 * place as G blocks of N rows against a [G, M, K] activation).  For every
 * group g:  y[g] = contraction(x[g], W[g*N .. g*N+N-1], b[g*N ..]) under
 * `spec`, exactly as poot_contract computes it.
 *   x [G, M, K], W [G*N, K], b [G*N] or NULL, y [G, M, N] (float32 when
 *   spec->out_f32), step operands [G*M, ld] (row g*M + m belongs to group g).
 * A batched contraction with one shared W is the plain call with M' = G*M.
 * G >= 1 with G*M and G*N at most 2^31 - 1; other errors as poot_contract.
 */
POOT_API int poot_contract_grouped(const void* x, const void* w, const void* b, void* y, int64_t G, int64_t M,
                                   int64_t N, int64_t K, const poot_contraction_spec* spec,
                                   const poot_linear_options* opts, poot_stream_t stream);

/*
 * Split-K without any allocation.  The pages have no counterpart to this
 * entry point: it is a library addition for callers that must not allocate
 * device memory — code that runs under a caching allocator holding the
 * device's memory budget (a library cudaMalloc there can fail or fragment
 * the pool), and serving loops with a fixed memory footprint that cannot
 * take an allocation's implicit device synchronisation.
 *
 * Computes y = FP16(x . W^T) + b on the GEMM (never the GEMV, whatever M)
 * exactly as poot_linear_f16_ex with gemm_split_k = split_k and the GEMM
 * variant for these pointers (GEMM_TMA when x and w are 16-byte aligned and
 * K % 8 == 0, else GEMM_CPASYNC when both are 4-byte aligned and K is even,
 * else GEMM_REG): same tile plan, same summation order, hence the same
 * bits.  The FP32 partial sums live in one device array compiled into the
 * library, POOT_NOALLOC_SCRATCH_BYTES per device, instead of the per-stream
 * workspace.
 * split_k: 2 .. 16 and must divide ceil(K / 64); split_k * M * N * 4 must
 *   not exceed POOT_NOALLOC_SCRATCH_BYTES.  Otherwise POOT_ERR_INVALID_ARG,
 *   before any CUDA call, with nothing queued.  K >= 1.
 * Other arguments, alignment, ownership and errors as poot_linear_f16.
 * The array needs no clearing: every element a call reads was written
 *   earlier in the same call.
 * Sharing: the array is one per device, used by every call of this entry
 *   point on that device (no other entry point touches it).  Calls whose
 *   work can overlap in time — on different streams with no event or
 *   synchronisation ordering them — race on it and give wrong results;
 *   calls on one stream, or otherwise ordered, are safe.
 * Setup: the first call on each device looks the array's address up
 *   (cudaGetSymbolAddress, with that device current) and keeps it; make
 *   that first call outside stream capture.
 */
#define POOT_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
POOT_API int poot_linear_f16_splitk_noalloc(const void* x, const void* w, const void* b, void* y, int64_t M,
                                            int64_t N, int64_t K, int split_k, poot_stream_t stream);

/* ---- Tensor-parallel linear -----------------------------------------------
 *
 * "The Graph IR", Primitive operations, the AllReduce / AllGather row
 * (tensor-parallel collectives; AllGather multiplies the gather axis by the
 * number of ranks), and "Model and Distributed IR", section "Boundary between
 * the layers" (linear(x, w) with a tensor-parallel strategy becomes
 * rank-local matmul tasks, a collective, and a reconstructed result that
 * equals the source semantics).  The collective itself is the caller's (NCCL
 * through torch.distributed in the Python binding); these are the host plan
 * and the device steps around it:
 *
 *   column split (over N): rank r holds W[begin_r:end_r, :] and b[begin_r:end_r]
 *     and computes y_r = poot_linear_f16(x, W_r, b_r) ([M, N_r], bit-identical
 *     to those columns of the one-GPU result); an all-gather puts every y_r
 *     in its slot; poot_linear_gather_columns assembles y [M, N].
 *   row split (over K): rank r holds x[:, begin_r:end_r] and
 *     W[:, begin_r:end_r] and computes the FP32 partial sums S_r with
 *     poot_contract (out_f32, no bias); an all-reduce adds them in FP32 (one
 *     legal summation order, rule 1 of the contract); poot_linear_f16_finish
 *     rounds once: y = RN16(RN16(S) + b).  Rounding or adding b per rank
 *     before the reduction would break the contract's rule 2.
 */

/*
 * Shard [*begin, *end) of rank `rank` among `world` ranks over an axis of
 * `extent` elements: contiguous ranges, every one but the last
 * ceil(extent / world) rounded up to a multiple of 8 wide (so a shard of a
 * 16-byte-aligned row-major operand stays 16-byte aligned), trailing ranks
 * possibly empty.  Pure host logic, no CUDA call.
 * Errors: POOT_ERR_INVALID_ARG for extent outside [0, 2^31), world outside
 * [1, 65536], rank outside [0, world), or a NULL output pointer.
 */
POOT_API int poot_linear_tp_shard(int64_t extent, int world, int rank, int64_t* begin, int64_t* end);

/*
 * y [M, N] (row-major binary16, device) from the column shards of a
 * tensor-parallel linear: slots (device) holds `world` slots of slot_elems
 * elements each, slot r holding rank r's y_r [M, N_r] row-major, its
 * columns [begin_r, end_r) as poot_linear_tp_shard(N, world, r) gives them.
 * A pure copy (bits unchanged), on `stream`, asynchronous.
 * slot_elems must hold the widest shard (M * N_0); y must not overlap the
 * slots.  Errors: POOT_ERR_INVALID_ARG (sizes, NULL, overlap),
 * POOT_ERR_MISALIGNED (a pointer not 2-byte aligned), POOT_ERR_CUDA.
 */
POOT_API int poot_linear_gather_columns(const void* slots, void* y, int64_t M, int64_t N, int world,
                                        int64_t slot_elems, poot_stream_t stream);

/*
 * y = RN16(RN16(S) + b) for an FP32 sum S [M, N] (device, row-major; the
 * all-reduced partial sums of a row split), b [N] and y [M, N] binary16
 * (device).  The epilogue of poot_linear_f16 applied to a given sum, on
 * `stream`, asynchronous.  S 4-byte aligned, b and y 2-byte aligned, y not
 * overlapping S or b.  Errors as poot_linear_gather_columns.
 */
POOT_API int poot_linear_f16_finish(const float* S, const void* b, void* y, int64_t M, int64_t N,
                                    poot_stream_t stream);

/* Library version, MAJOR * 10000 + MINOR * 100 + PATCH. */
POOT_API int poot_linear_version(void);

#ifdef __cplusplus
}
#endif

#endif /* POOT_LINEAR_H */
