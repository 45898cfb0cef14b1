/*
 * olc_matmul.h -- C ABI of the GB300 ONNX MatMul library (libolc_matmul.so).
 *
 * The operator is ONNX MatMul: vector, matrix and batched matrix products with
 * NumPy-style batch broadcasting ("MatMul Kernel Design", introduction and
 * section "Shape and plan model").  A plan is built once from the two operand
 * shapes and the element type; executing it enqueues CUDA kernels on the
 * caller's stream.
 *
 * Conventions shared by every entry point
 *  - Tensors are dense and row-major (C-contiguous).  A, B and Y are device
 *    pointers owned by the caller; the library never frees them.
 *  - A and B have the same element type (olc_dtype); Y has it too.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Execution is asynchronous: a return of OLC_OK means the work
 *    was enqueued.
 *  - Every shape or type error is reported by olc_matmul_plan_create, before
 *    any device work ("Types and algorithm selection": dynamic negative
 *    dimensions, mixed or unsupported types and incompatible matrix or batch
 *    dimensions fail before compute).
 *  - Functions returning olc_status never abort the process.
 *  - A plan is bound to the CUDA device that was current when it was created.
 *    It may be executed on any stream of that device; its calls must not run
 *    concurrently from two host threads.  Executes that use the plan's own
 *    device state -- its workspace (olc_matmul_plan_workspace_bytes > 0:
 *    split reductions, the per-call transpose of an 8-bit B) or its staging
 *    buffer (olc_matmul_plan_staging_copies > 0) -- are ordered across
 *    streams by the plan: such an execute on another stream than the
 *    previous one waits, on the GPU, for that previous one to finish
 *    (cudaStreamWaitEvent on an event the plan records; one event, created
 *    at the first such execute).  While a stream is capturing a graph the
 *    plan records and waits for nothing: ordering captured launches against
 *    other uses of the plan is the caller's.
 */
#ifndef OLC_MATMUL_H
#define OLC_MATMUL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types, numbered as ONNX TensorProto data types.  FLOAT and DOUBLE
 * accumulate natively; FLOAT16 and BFLOAT16 accumulate in float32 and narrow
 * the result once with round-to-nearest-even ("Types and algorithm
 * selection"; "Gemm and MatMul Performance Roadmap", section "Scope and type
 * matrix").  The 8-bit float operand types ("Gemm and MatMul Performance
 * Roadmap", the Float8 packing-format item) decode exactly to float32,
 * accumulate in float32, and give a FLOAT output (4 bytes per element): A
 * and B have the 8-bit type, Y (and a fused residual) is float32.  They are
 * MatMul types only (Gemm plans reject them).  E4M3FN and E5M2 run on the
 * tensor cores: tcgen05 kind::f8f6f4 tiles for general shapes, and the
 * warp-level mma.sync m16n8k32 for few rows (SKINNY_M from 4 rows), few
 * columns (SKINNY_N up to 8) and small outputs over a long K (SPLIT_K); the
 * FNUZ variants, whose encodings the tensor cores do not take, always run on
 * SIMT decode kernels (SKINNY_M, GENERAL_SIMT, DIRECT). */
typedef enum {
    OLC_FLOAT = 1,
    OLC_FLOAT16 = 10,
    OLC_DOUBLE = 11,
    OLC_BFLOAT16 = 16,
    OLC_FLOAT8E4M3FN = 17,   /* 1-4-3, bias 7, no infinities, S.1111.111 NaN */
    OLC_FLOAT8E4M3FNUZ = 18, /* 1-4-3, bias 8, no infinities, no -0, 0x80 NaN */
    OLC_FLOAT8E5M2 = 19,     /* 1-5-2, bias 15, IEEE-style infinities / NaNs */
    OLC_FLOAT8E5M2FNUZ = 20  /* 1-5-2, bias 16, no infinities, no -0, 0x80 NaN */
} olc_dtype;

typedef enum {
    OLC_OK = 0,
    OLC_ERR_NULL = 1,             /* a required pointer argument is NULL           */
    OLC_ERR_RANK = 2,             /* rank 0, or rank above OLC_MAX_RANK            */
    OLC_ERR_NEGATIVE_DIM = 3,     /* a dimension is negative                       */
    OLC_ERR_K_MISMATCH = 4,       /* A's last dim differs from B's contraction dim */
    OLC_ERR_BATCH_MISMATCH = 5,   /* batch extents neither equal nor 1             */
    OLC_ERR_DTYPE = 6,            /* element type not supported                    */
    OLC_ERR_ALIGNMENT = 7,        /* a forced algorithm cannot take these shapes   */
    OLC_ERR_BUFFER_TOO_SMALL = 8, /* a checked execute got a buffer too small      */
    OLC_ERR_NO_CONSTANT_B = 9,    /* a B-less execute on a plan that owns no B     */
    OLC_ERR_CUDA = 10,            /* a CUDA runtime call failed                    */
    OLC_ERR_DEVICE_TIMEOUT = 11,  /* a bounded device-side wait ran out            */
    OLC_ERR_OOM = 12,             /* workspace allocation failed                   */
    OLC_ERR_INVALID = 13,         /* an argument is out of its documented range    */
    OLC_ERR_WRONG_DEVICE = 14,    /* current device differs from the plan or stream */
    OLC_ERR_SCRATCH_LIMIT = 15,   /* needs more than the static scratch array      */
    OLC_ERR_NEEDS_RESIDUAL = 16   /* the plan fuses a residual: use the fused call */
} olc_status;

/* Activation of the fused epilogue (applied after bias and residual, before
 * narrowing).  GELU is the exact form x * Phi(x) = x / 2 * (1 + erf(x / sqrt 2)). */
typedef enum {
    OLC_ACT_NONE = 0,
    OLC_ACT_RELU = 1,             /* max(x, 0); NaN stays NaN                      */
    OLC_ACT_GELU = 2
} olc_activation;

/* The algorithm a plan runs ("MatMul Kernel Design", section "Types and
 * algorithm selection": direct execution for small reductions, skinny-M or
 * skinny-N kernels when one output dimension underfills the ordinary tile,
 * split-K for the tiny-output long-reduction corner, the general tiled engine
 * otherwise).  EMPTY and ZERO_FILL cover outputs with no elements and K == 0. */
typedef enum {
    OLC_ALGO_AUTO = -1,       /* only as an argument: restore automatic choice */
    OLC_ALGO_EMPTY = 0,       /* output has no elements: nothing is launched    */
    OLC_ALGO_ZERO_FILL = 1,   /* K == 0: Y is set to zero, A and B are not read */
    OLC_ALGO_DIRECT = 2,      /* small SIMT tile kernel, any shape or alignment */
    OLC_ALGO_SKINNY_M = 3,    /* M <= 16: stream B once, vectorised along N     */
    OLC_ALGO_SKINNY_N = 4,    /* N <= 16: stream A once, vectorised along K     */
    OLC_ALGO_SPLIT_K = 5,     /* K partitioned, fixed-order reduction           */
    OLC_ALGO_GENERAL_TC = 6,  /* FLOAT16/BFLOAT16: tcgen05 tensor-core tiles    */
    OLC_ALGO_GENERAL_SIMT = 7 /* FLOAT/DOUBLE: FFMA / DFMA register tiles       */
} olc_algorithm;

#define OLC_MAX_RANK 8

typedef struct olc_matmul_plan olc_matmul_plan;

/*
 * Build a plan for Y = MatMul(A, B).
 *
 * "MatMul Kernel Design", section "Shape and plan model": the plan resolves
 * the complete output shape before execution -- a rank-one A [K] is promoted
 * to [1, K] and a rank-one B [K] to [K, 1] and the promoted dimension is
 * squeezed from the output; the leading batch dimensions are broadcast
 * multidirectionally (aligned on the right; equal, or one side 1); each
 * operand gets per-dimension batch strides in elements, 0 where it is
 * broadcast; then one GEMM is planned per broadcast batch item ("Gemm and
 * MatMul Performance Roadmap", section "Phase 4: complete MatMul", steps 1-6,
 * including the collapse of contiguous batch dimensions).
 *
 *  a_shape[a_rank], b_shape[b_rank]: operand shapes, 1 <= rank <= OLC_MAX_RANK.
 *      An extent 0 is allowed; it broadcasts against 1 (giving 0) and is an
 *      error against an extent > 1.
 *  dtype: the common element type of A, B and Y.
 *  out: receives the new plan (owned by the caller; free with
 *      olc_matmul_plan_destroy).  Set to NULL on error.
 *
 * Errors: OLC_ERR_NULL, OLC_ERR_RANK, OLC_ERR_NEGATIVE_DIM, OLC_ERR_K_MISMATCH,
 * OLC_ERR_BATCH_MISMATCH, OLC_ERR_DTYPE, OLC_ERR_INVALID (A, B or Y would
 * hold more than 2^62 bytes, so that element offsets could overflow int64),
 * OLC_ERR_OOM (host or workspace allocation), OLC_ERR_CUDA.  If a CUDA
 * device is present and the chosen
 * algorithm needs a split reduction workspace, it is allocated here
 * (cudaMalloc on the current device) and owned by the plan.
 */
olc_status olc_matmul_plan_create(const int64_t* a_shape, int a_rank,
                                  const int64_t* b_shape, int b_rank,
                                  olc_dtype dtype, olc_matmul_plan** out);

/* Free a plan and its workspace.  NULL is accepted.  The caller must make sure
 * no execute of this plan is still running on the device. */
void olc_matmul_plan_destroy(olc_matmul_plan* plan);

/*
 * Enqueue Y = MatMul(A, B) on `stream`.
 *
 * "MatMul Kernel Design", sections "Shape and plan model" and "Scheduling
 * and invariants": one GEMM per broadcast batch item, run as one launch over
 * all items (the batch index is part of the grid); broadcast operands are read
 * through zero batch strides, never copied.  Y must hold every batch item's
 * complete M x N matrix: prod(output shape) elements.
 *
 *  A: prod(a_shape) elements, B: prod(b_shape) elements, Y: prod(out shape)
 *     elements, all device pointers of the plan's dtype.
 *  An output with no elements returns OLC_OK without launching anything and
 *     without reading A, B or Y (they may be NULL).  With K == 0 and a
 *     non-empty output, Y is filled with zeros and A and B are not read.
 *  Alignment: FLOAT16 / BFLOAT16 products stay on the tensor cores for any
 *     2-byte aligned pointers and any N and K.  An operand the kernels
 *     cannot read in place (pointer off a 16-byte boundary; on the general
 *     tiles, stored rows that are not a multiple of 16 bytes) is first
 *     copied by a kernel of this library into a staging buffer the plan
 *     owns: allocated (cudaMalloc) at olc_matmul_plan_create when the shape
 *     alone needs it, otherwise at the first execute that does -- make that
 *     first call before any stream capture.  The general tiles store a Y of
 *     any alignment; skinny and split-K products with a misaligned Y (or
 *     residual) run on the general tiles.  FLOAT, DOUBLE and the 8-bit
 *     types need 16-byte aligned A, B and Y on their skinny, split-K and
 *     tensor-core paths and run the DIRECT kernel otherwise.
 *     olc_matmul_plan_algorithm_for / _staging_copies report the route.
 *
 * Errors: OLC_ERR_NULL (plan, or a data pointer of a non-empty product),
 * OLC_ERR_INVALID (a pointer not aligned to its element size),
 * OLC_ERR_WRONG_DEVICE, OLC_ERR_CUDA (a launch failed), OLC_ERR_OOM (a
 * staging buffer could not be allocated).
 * Device-side failures are not seen here; use olc_matmul_execute_checked.
 */
olc_status olc_matmul_execute(const olc_matmul_plan* plan, const void* A, const void* B,
                              void* Y, void* stream);

/*
 * olc_matmul_execute plus validation of the buffer sizes ("Scheduling and
 * invariants": the output buffer must cover every broadcast batch item and
 * its complete M x N matrix), then a synchronisation of `stream` and a read of
 * the device error word that the library's bounded waits set.
 *
 *  a_numel, b_numel, y_numel: elements available behind A, B and Y.
 * Errors: as olc_matmul_execute, plus OLC_ERR_BUFFER_TOO_SMALL (before any
 * launch) and OLC_ERR_DEVICE_TIMEOUT (a kernel gave up waiting; Y is then
 * unspecified).  The device error word is cleared by this call.
 */
olc_status olc_matmul_execute_checked(const olc_matmul_plan* plan,
                                      const void* A, int64_t a_numel,
                                      const void* B, int64_t b_numel,
                                      void* Y, int64_t y_numel, void* stream);

/*
 * The same product from host buffers: copies A and B from host memory into
 * the caller's device buffers, runs the plan, and copies Y back, ordered on
 * `stream` (use pinned host memory for asynchronous copies).  A_host/B_host/
 * Y_host: host pointers; A_dev/B_dev/Y_dev: device buffers of the same sizes.
 * Returns after enqueueing; synchronise `stream` before reading Y_host.
 * A single 2-D product (a batch folded into rows) of at least 4096 rows on
 * the general kernels, without a residual, runs as a pipeline over four row
 * chunks: B and the A chunks are copied in on one internal stream, chunk i
 * is computed on `stream` once its rows have arrived, and its rows of Y are
 * copied out on a second internal stream while later chunks compute; the
 * call's work still starts after earlier work on `stream` and later work on
 * `stream` starts after the last copy.  The two streams and the events are
 * created (and owned by the plan) at the first such call; nothing else is
 * allocated.  Other products: the three steps in order on `stream`.  A plan
 * must not run two host-buffer executes at once on different streams.
 * Errors: as olc_matmul_execute.
 */
olc_status olc_matmul_execute_host(const olc_matmul_plan* plan,
                                   const void* A_host, const void* B_host, void* Y_host,
                                   void* A_dev, void* B_dev, void* Y_dev, void* stream);

/* ---- the Gemm operator ------------------------------------------------- */

/*
 * Build a plan for ONNX Gemm: Y = alpha * A' B' + beta * C, on the same GEMM
 * engine ("Gemm and MatMul Performance Roadmap", section "Scope and type
 * matrix": Gemm handles rank-2 inputs, alpha, beta, an optional broadcast
 * bias and transA / transB).
 *
 *  a_shape[2]: A as stored: [M, K], or [K, M] with trans_a != 0.
 *  b_shape[2]: B as stored: [K, N], or [N, K] with trans_b != 0.
 *  alpha, beta: scalars (applied in the accumulator type: float32 for FLOAT,
 *      FLOAT16, BFLOAT16; float64 for DOUBLE).
 *  c_shape[c_rank]: C's shape, unidirectionally broadcast to [M, N]: rank 0
 *      (scalar), [N], [1, N], [M, 1], [M, N] ...; c_rank = -1: no C (the bias
 *      term is absent and beta is unused).
 *  dtype: the element type of A, B, C and Y.
 * Y is [M, N].  FLOAT16 / BFLOAT16 accumulate in float32, apply the
 * epilogue in float32 and narrow once.  With K == 0, Y = beta * C.
 * Errors: OLC_ERR_NULL, OLC_ERR_RANK (c_rank outside -1..2),
 * OLC_ERR_NEGATIVE_DIM, OLC_ERR_K_MISMATCH, OLC_ERR_BATCH_MISMATCH (C does
 * not broadcast to [M, N]), OLC_ERR_DTYPE, OLC_ERR_INVALID (A, B or Y would
 * hold more than 2^62 bytes), OLC_ERR_OOM, OLC_ERR_CUDA.
 * Free with olc_matmul_plan_destroy; the query functions below apply.
 */
olc_status olc_gemm_plan_create(const int64_t* a_shape, const int64_t* b_shape, int trans_a,
                                int trans_b, double alpha, double beta, const int64_t* c_shape,
                                int c_rank, olc_dtype dtype, olc_matmul_plan** out);

/*
 * Enqueue the Gemm on `stream`.  A, B, C, Y: device pointers of the plan's
 * dtype, dense row-major as described at creation (C may be NULL only if the
 * plan has no C).  The same execution rules as olc_matmul_execute.
 * Errors: OLC_ERR_NULL, OLC_ERR_WRONG_DEVICE, OLC_ERR_CUDA, OLC_ERR_OOM.
 */
olc_status olc_gemm_execute(const olc_matmul_plan* plan, const void* A, const void* B,
                            const void* C, void* Y, void* stream);

/* ---- plan-owned constant B ---------------------------------------------- */

/*
 * Give the plan its own copy of a constant B ("MatMul Kernel Design",
 * section "Shape and plan model": the library plan can own a constant B with
 * a lifetime independent of the source buffer; section "Scheduling and
 * invariants": the constant-B storage must contain exactly the planned
 * matrix).  B: host or device pointer to b_numel elements of the plan's
 * dtype, laid out as planned (for Gemm, as stored: [K, N] or [N, K]); the
 * copy is made on `stream` and has completed when the call returns, so the
 * caller may free or overwrite its buffer.  Device memory is allocated once
 * (cudaMalloc on the plan's device) and freed with the plan; calling again
 * replaces the contents.  The 16-bit and wider kernels read B's layout
 * directly.  A plan with 8-bit float operands on the tensor cores also keeps
 * B transposed ([N, K] bytes, the K-major operand the MMA reads; b_numel more
 * bytes of device memory), so executes with the constant B skip the
 * transpose that an execute with a caller's B runs first.  An 8-bit few-row
 * plan (SKINNY_M, E4M3FN / E5M2, 2 to 16 rows, one item, N and K multiples
 * of 16, kernel family automatic or 3) keeps the transposed B as well and from then on runs the
 * tcgen05 few-row kernel, which streams that copy straight to the MMA
 * (executes with a caller's B on such a plan run the same kernel, which then
 * transposes B in shared memory on the way).  Likewise a
 * FLOAT16 / BFLOAT16 plan on the general tensor-core tiles whose B rows are
 * not a multiple of 16 bytes (N not a multiple of 8) keeps B with rows
 * padded to 8 elements, so executes with the constant B copy nothing.
 * Errors:
 * OLC_ERR_NULL, OLC_ERR_BUFFER_TOO_SMALL (b_numel is not the planned size),
 * OLC_ERR_WRONG_DEVICE, OLC_ERR_OOM, OLC_ERR_CUDA.
 */
olc_status olc_matmul_plan_set_constant_b(olc_matmul_plan* plan, const void* B, int64_t b_numel,
                                          void* stream);

/* 1 if the plan owns a constant B, 0 otherwise (also for NULL). */
int olc_matmul_plan_has_constant_b(const olc_matmul_plan* plan);

/* Y = MatMul(A, B) with the plan-owned B.  Rejected with OLC_ERR_NO_CONSTANT_B
 * when the plan owns no B ("Scheduling and invariants": the constant-only
 * Execute is rejected when the plan does not own B).  Otherwise as
 * olc_matmul_execute. */
olc_status olc_matmul_execute_constant(const olc_matmul_plan* plan, const void* A, void* Y,
                                       void* stream);

/* The Gemm with the plan-owned B; as olc_gemm_execute otherwise. */
olc_status olc_gemm_execute_constant(const olc_matmul_plan* plan, const void* A, const void* C,
                                     void* Y, void* stream);

/* ---- fused epilogue ----------------------------------------------------- */

/*
 * Fuse elementwise work into the product's store ("Gemm and MatMul
 * Performance Roadmap", the fused-epilogue row of its opportunity table and
 * the broadcast / fused epilogue item of its plan: bias, residual, activation
 * and output conversion in one typed epilogue, with no intermediate tensor).
 * Per output element, in the accumulator type (float32 for FP16/BF16/FP32,
 * float64 for FP64), each step rounded on its own:
 *     v = alpha * acc + beta * C      (Gemm plans; acc for MatMul plans)
 *     v = v + R                       (residual != 0)
 *     v = act(v)                      (activation, olc_activation)
 * then v is narrowed to the output type once.  R has the output's shape,
 * dtype and dense row-major layout (the full broadcast output for batched
 * MatMul plans).  activation: OLC_ACT_NONE / RELU / GELU; residual: 0 or 1.
 * Errors: OLC_ERR_NULL, OLC_ERR_INVALID (value out of range).  A plan with a
 * residual must be run through olc_matmul_execute_fused; the other execute
 * calls return OLC_ERR_NEEDS_RESIDUAL for it.  An activation alone applies
 * to every execute call.
 */
olc_status olc_matmul_plan_set_epilogue(olc_matmul_plan* plan, int activation, int residual);

/*
 * Execute with the fused epilogue.  B: device pointer, or NULL to use the
 * plan-owned constant B (OLC_ERR_NO_CONSTANT_B when the plan owns none).
 * C: the Gemm bias (required when the Gemm plan has one, ignored otherwise).
 * R: residual, device pointer, required when the plan fuses a residual
 * (OLC_ERR_NULL otherwise); it may not overlap Y unless R == Y exactly
 * (each element's residual is read by the thread that then writes it).
 * Pointers the fast kernels read with 16-byte vectors (A, B, Y, R) that are
 * not 16-byte aligned send the product to the DIRECT kernel.  Asynchronous
 * on `stream`, as olc_matmul_execute.
 */
olc_status olc_matmul_execute_fused(const olc_matmul_plan* plan, const void* A, const void* B,
                                    const void* C, const void* R, void* Y, void* stream);

/* ---- grouped products ---------------------------------------------------- */

/*
 * Many independent rank-2 products in one launch ("Gemm and MatMul
 * Performance Roadmap": the batch-fusion row of its opportunity table, for
 * hundreds of tiny or irregular products, and the GroupedGemm interface of
 * its plan).  Member i computes Y_i[m_i, n_i] = A_i[m_i, k_i] @ B_i[k_i, n_i],
 * all row-major and dense, accumulated as MatMul accumulates (float32 for
 * FLOAT16 / BFLOAT16 / FLOAT, float64 for DOUBLE) and narrowed once.
 */
typedef struct olc_grouped_plan olc_grouped_plan;

/* m, n, k: host arrays of `count` dimensions (copied; the caller keeps
 * ownership).  Errors: OLC_ERR_NULL, OLC_ERR_INVALID (count <= 0, a
 * member's A, B or Y above 2^62 bytes, or more than 2^31 - 1 output tiles of
 * 64 x 64 in all), OLC_ERR_NEGATIVE_DIM, OLC_ERR_DTYPE, OLC_ERR_OOM. */
olc_status olc_grouped_plan_create(int count, const int64_t* m, const int64_t* n, const int64_t* k,
                                   olc_dtype dtype, olc_grouped_plan** out);

/* NULL is accepted. */
void olc_grouped_plan_destroy(olc_grouped_plan* plan);

/* Output tiles (64 x 64) of all members, and the member count; -1 for NULL. */
int64_t olc_grouped_plan_tiles(const olc_grouped_plan* plan);
int olc_grouped_plan_count(const olc_grouped_plan* plan);

/*
 * Run the group: A, B, Y are DEVICE arrays of `count` device pointers (member
 * i's operands and output).  One launch on `stream`; returns after enqueueing.
 * The first call on a device copies the plan's descriptor table there
 * (cudaMalloc, freed with the plan); later calls allocate nothing.  Members
 * with an empty output are skipped (their pointers may be NULL); K == 0
 * members get zeros.  Errors: OLC_ERR_NULL, OLC_ERR_WRONG_DEVICE, OLC_ERR_OOM,
 * OLC_ERR_CUDA.
 */
olc_status olc_grouped_execute(const olc_grouped_plan* plan, const void* const* A, const void* const* B,
                               void* const* Y, void* stream);

/* ---- queries ----------------------------------------------------------- */

/* Output shape: writes up to `capacity` extents into shape[] and the rank
 * into *rank (0 = a scalar with one element, from two rank-one operands).
 * Errors: OLC_ERR_NULL, OLC_ERR_INVALID (capacity too small). */
olc_status olc_matmul_plan_output_shape(const olc_matmul_plan* plan, int64_t* shape,
                                        int capacity, int* rank);

/* Promoted matrix sizes and the number of broadcast batch items, before any
 * folding: the product is batch x ([M, K] @ [K, N]).  NULL outputs skipped. */
olc_status olc_matmul_plan_dims(const olc_matmul_plan* plan, int64_t* M, int64_t* N,
                                int64_t* K, int64_t* batch);

/* The broadcast batch shape (rank *batch_rank) and each operand's batch
 * strides in elements, 0 where the operand is broadcast ("each input receives
 * precomputed batch strides, including zero strides for broadcast
 * dimensions").  Arrays need OLC_MAX_RANK entries; NULL arrays skipped. */
olc_status olc_matmul_plan_batch(const olc_matmul_plan* plan, int* batch_rank,
                                 int64_t* batch_shape, int64_t* a_strides,
                                 int64_t* b_strides);

/* The launch geometry after batch collapse and folding: GEMM rows M' (M times
 * the folded batch), the number of batch items one launch walks, and the
 * number of collapsed batch dimensions.  NULL outputs skipped. */
olc_status olc_matmul_plan_launch_shape(const olc_matmul_plan* plan, int64_t* rows,
                                        int64_t* items, int* collapsed_rank);

/* Selected algorithm (an olc_algorithm value), or -1 for a NULL plan. */
int olc_matmul_plan_algorithm(const olc_matmul_plan* plan);

/* The algorithm an execute with these pointers runs (R: the fused
 * residual, or NULL), or -1 for a NULL plan.  It differs from the plan's
 * algorithm only for pointers off a 16-byte boundary: FLOAT16 / BFLOAT16
 * skinny and split-K products whose Y (or R) is misaligned run on the
 * general tensor-core tiles, and other types' products with any misaligned
 * pointer run on DIRECT.  Host only; nothing is launched. */
int olc_matmul_plan_algorithm_for(const olc_matmul_plan* plan, const void* A, const void* B,
                                  const void* Y, const void* R);

/* Staging copies (0, 1 or 2) an execute with these pointers makes before its
 * product kernel, or -1 for a NULL plan.  FLOAT16 / BFLOAT16 products on the
 * tensor cores copy an operand the kernels cannot read in place: one whose
 * pointer is off a 16-byte boundary, and, on the general tiles, one whose
 * stored rows are not a multiple of 16 bytes (K or N not a multiple of 8) --
 * into rows padded to 8 elements that the tiles read through a row pitch.
 * Host only; nothing is launched. */
int olc_matmul_plan_staging_copies(const olc_matmul_plan* plan, const void* A, const void* B,
                                   const void* Y, const void* R);

/* Force an algorithm (testing and tuning sweeps); OLC_ALGO_AUTO restores the
 * automatic choice.  Errors: OLC_ERR_NULL, OLC_ERR_INVALID (unknown value),
 * OLC_ERR_ALIGNMENT (the algorithm cannot take this shape or type),
 * OLC_ERR_OOM / OLC_ERR_CUDA (workspace).  EMPTY and ZERO_FILL plans accept
 * only themselves or AUTO. */
olc_status olc_matmul_plan_force_algorithm(olc_matmul_plan* plan, int algo);

/* Tuning override of the number of K slices of SPLIT_K and SKINNY_M plans,
 * and of FLOAT GENERAL_SIMT plans (which slice K when their 128 x 128 tiles
 * are fewer than the SMs; 1 = never) (0 = automatic choice from the SM count;
 * values are clamped to what the shape allows).  Re-sizes the workspace.  Errors: OLC_ERR_NULL,
 * OLC_ERR_INVALID (negative or above 4096), OLC_ERR_OOM, OLC_ERR_CUDA. */
olc_status olc_matmul_plan_set_splits(olc_matmul_plan* plan, int splits);

/* K slices the plan currently uses (1 when it does not split). */
int olc_matmul_plan_splits(const olc_matmul_plan* plan);

/* Tuning override of the kernel family.  GENERAL_TC plans: 0 = automatic
 * (FLOAT16 / BFLOAT16: when the 128 x 256 tiles would fill at most half the
 * SMs, the cluster split-K -- the K blocks of each tile cut into slices run
 * by the CTAs of one thread-block cluster, whose float32 partial tiles meet
 * in the plan's workspace and are summed in slice order, so the result does
 * not depend on timing; otherwise CTA pairs whenever N >= 256), 1 = one CTA
 * per 128 x 256 output tile, 2 = pairs of CTAs on one TPC sharing a 256 x
 * 256 tile (tcgen05 cta_group::2).  SKINNY_N plans of
 * FLOAT16 / BFLOAT16: 0 = automatic, 1 = the tcgen05 16-column kernel,
 * 2 = the register-streaming mma.sync kernel wherever it applies (one B for
 * all rows, K a multiple of 8, B^T within its shared-memory budget).
 * SKINNY_M plans of FLOAT16 / BFLOAT16: 0 = automatic (tensor cores from 4
 * rows, or from 2 rows with a B of 256 MB or more), 1 = the SIMT streaming
 * kernel, 2 = the swapped-operand tcgen05 kernel.  SKINNY_M plans of
 * FLOAT8E4M3FN / FLOAT8E5M2: 0 = automatic (the warp-level MMA kernel from 4
 * rows), 1 = the SIMT streaming kernel, 2 = the warp-level MMA kernel
 * (mma.sync m16n8k32 on B fragments transposed in registers), 3 = the
 * tcgen05 kernel with swapped operands (kind::f8f6f4, 128 output columns per
 * MMA; B transposed in shared memory, or read transposed from the plan's
 * constant B; one item, N and K multiples of 16, else the warp-level MMA
 * kernel).  GENERAL_TC
 * plans of 8-bit floats: 1 = one CTA per 128 x 256 tile instead of CTA pairs.
 * Results are identical within the parity tolerance either way (the
 * variants sum K in different orders only where one splits it).  Errors:
 * OLC_ERR_NULL, OLC_ERR_INVALID. */
olc_status olc_matmul_plan_set_tc_variant(olc_matmul_plan* plan, int variant);

/* Kernel launches one execute of this plan makes with 16-byte aligned
 * pointers (0 for EMPTY): the product kernel, plus the staging copies its
 * shape needs (FLOAT16 / BFLOAT16 on the general tiles with K or N not a
 * multiple of 8; none for a B kept padded with the plan's constant B), plus
 * the B transpose of 8-bit tensor-core plans without a constant B. */
int olc_matmul_plan_launches(const olc_matmul_plan* plan);

/* Bytes of device workspace the plan owns for split reductions (SPLIT_K,
 * SKINNY_M and SKINNY_N slices, the FLOAT register tiles' K slices, the
 * general FP16 / BF16 tiles' cluster split-K) and the FP8 B transpose, 0 if
 * none; staging buffers are not included. */
size_t olc_matmul_plan_workspace_bytes(const olc_matmul_plan* plan);

/* One-line description of the plan (algorithm, type, shape after batch
 * collapse and fold, K slices, the cluster split-K's slices where the general
 * FP16 / BF16 tiles use it, workspace bytes, SM count) written into buf
 * (NUL-terminated, truncated to cap).  Returns the full length. */
int olc_matmul_plan_describe(const olc_matmul_plan* plan, char* buf, size_t cap);

/* Static strings; never NULL. */
const char* olc_status_string(int status);
const char* olc_algorithm_name(int algo);

/* Library version, as major * 10000 + minor * 100 + patch. */
int olc_version(void);

/* ---- testing hooks ------------------------------------------------------ */

/* The 64-bit shared-memory matrix descriptor and the 32-bit instruction
 * descriptor the tensor-core kernel hands to tcgen05.mma (PTX ISA, tcgen05
 * "shared memory descriptor" and "instruction descriptor" for kind::f16),
 * exported so a host test can check the bit layout.  Pure functions. */
uint64_t olc_debug_tc_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout);
uint32_t olc_debug_tc_instr_desc(int is_bf16, int m, int n, int a_mn_major, int b_mn_major);

/* Testing hook: the tcgen05 kind::f8f6f4 instruction descriptor the FP8
 * kernel uses (fmt 0 = E4M3, 1 = E5M2; both operands K-major; float32
 * accumulator).  Host only, no device needed. */
uint32_t olc_debug_f8_instr_desc(int fmt, int m, int n);

/* Self-test of the bounded device-side wait the tensor-core kernel uses on
 * every mbarrier: one thread waits for an mbarrier phase that completes only
 * if `arrive` is non-zero, giving up after `limit_ns` nanoseconds of
 * %globaltimer.  Synchronises `stream`.  Returns OLC_OK when the wait
 * succeeded and OLC_ERR_DEVICE_TIMEOUT when it ran out (the device error word
 * is read and cleared); the CUDA context stays usable either way. */
olc_status olc_debug_wait_selftest(uint64_t limit_ns, int arrive, void* stream);

/* Measurement hook: the arithmetic rate the FP32 / FP64 pipes deliver on the
 * current device (the FLOAT and DOUBLE kernels keep native precision, so
 * their roofline is the FMA pipes, not the tensor cores or memory).  Runs
 * SM count x 4 blocks of 256 threads, each thread `iters` iterations of
 * independent FMA chains with no memory traffic, timed with CUDA events on
 * `stream` (synchronised); *flops receives flop/s (an FMA counts 2).
 * kind: 0 = paired FP32 FMA (fma.rn.f32x2), 1 = FP32 FMA, 2 = FP64 FMA,
 * 3 = FP64 tensor-core MMA (mma.sync m8n8k4 .f64).  Errors: OLC_ERR_NULL,
 * OLC_ERR_INVALID (kind outside 0..3, iters outside 1..2^40), OLC_ERR_CUDA. */
olc_status olc_debug_alu_rate(int kind, int64_t iters, void* stream, double* flops);

/* ---- allocation-free split-K ------------------------------------------- */

/* Size of the device array behind olc_matmul_split_k_static: 4 MiB, held by
 * every GPU that loads this library until the process exits. */
#define OLC_SPLIT_K_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * Split-K product Y[M, N] = A[M, K] @ B[K, N] (dense row-major device
 * buffers, one element type) that allocates nothing.  The pages have no
 * counterpart for this entry point: it exists for callers that must not
 * allocate device memory while they run, such as a host framework whose
 * memory pool owns the whole device and forbids raw cudaMalloc, or a
 * latency-bound serving loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  The plan path allocates its split-K workspace with
 * cudaMalloc at olc_matmul_plan_create; this entry point instead keeps the
 * partial tiles and arrival counters in one file-scope device array of
 * OLC_SPLIT_K_STATIC_SCRATCH_BYTES bytes inside the library.
 *
 * It runs the SIMT split-K kernel (the plan path's kernel for FLOAT and
 * DOUBLE: partials per K slice, summed by the last-arriving block in slice
 * order) for every type, with the number of slices capped so the partials
 * fit the array (the plan path, by contrast, runs FLOAT16 / BFLOAT16 split-K
 * products on the tensor cores; on [32, 131072] x [131072, 32] FLOAT16 this
 * entry point takes about ten times as long).
 *
 *  dtype: OLC_FLOAT, OLC_DOUBLE, OLC_FLOAT16 or OLC_BFLOAT16.
 *  A, B, Y: caller-owned device pointers (M*K, K*N and M*N elements).
 *  M, N, K >= 0.  M*N == 0 returns OLC_OK with nothing launched; K == 0
 *  fills Y with zeros.
 *  stream: cudaStream_t as void* (NULL = legacy default stream).
 *
 * `stream` must belong to the current device (OLC_ERR_WRONG_DEVICE
 * otherwise): the array's address and the SM count are the current
 * device's.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress) and caches it.  Under CUDA's default lazy
 * module loading that lookup (or any earlier split-K launch of this
 * library) is also what loads the library's split-K module onto the device,
 * and with it the array: so the first call itself commits the 4 MiB of
 * device memory, and fails with OLC_ERR_CUDA if nothing is left.  Make that
 * first call at set-up time -- before a memory pool takes the rest of the
 * device, and before any stream capture on that device; later calls
 * allocate nothing.  Every call clears the arrival counters
 * with cudaMemsetAsync on `stream` before its kernel, so a call never depends
 * on what the previous one left in the array; but all calls share the one
 * array, so calls whose executions overlap on the GPU (other streams, other
 * host threads) race and must be serialised by the caller.
 *
 * Layout of the array: the first 16 KiB hold up to 4096 arrival counters,
 * the rest holds the partial tiles (32 x 32 accumulators per output tile and
 * K slice).  So ceil(M/32) * ceil(N/32) may be at most 1020 for FLOAT,
 * FLOAT16 and BFLOAT16 (float32 partials) and at most 510 for DOUBLE.
 *
 * Errors: OLC_ERR_DTYPE, OLC_ERR_NULL (a pointer of a non-empty product),
 * OLC_ERR_NEGATIVE_DIM, OLC_ERR_SCRATCH_LIMIT (more output tiles than the
 * limits above), OLC_ERR_WRONG_DEVICE (`stream` belongs to another device
 * than the current one), OLC_ERR_CUDA (the address lookup, memset or
 * launch failed).
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
olc_status olc_matmul_split_k_static(olc_dtype dtype, const void* A, const void* B, void* Y,
                                     int64_t M, int64_t N, int64_t K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OLC_MATMUL_H */
