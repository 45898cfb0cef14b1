// Internal interface between the host plan (api.cpp) and the kernel files.
// Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "olc_matmul.h"

namespace olc {

constexpr int kMaxBatchRank = OLC_MAX_RANK;

// Output batch item -> operand element offsets.  `dims` are the collapsed
// batch extents (outermost first); an operand's stride is 0 along a dimension
// it broadcasts.  The output itself is dense: item z starts at z * M * N.
struct BatchMap {
    int rank;
    int64_t dims[kMaxBatchRank];
    int64_t a_stride[kMaxBatchRank];
    int64_t b_stride[kMaxBatchRank];
};

// Gemm epilogue: y = alpha * acc + beta * C[i * c_rs + j * c_cs] (C of the
// output type, strides 0 along broadcast dimensions).  mode 0 = plain
// product (y = acc, MatMul), 1 = alpha/beta/C applied.  C may be NULL (no
// bias term).
struct Epilogue {
    int mode;                  // 0: Y = acc; 1: the steps below
    float alpha_f, beta_f;
    double alpha_d, beta_d;
    const void* C;             // bias, broadcast through (c_rs, c_cs); may be null
    int64_t c_rs, c_cs;
    const void* R;             // residual in Y's layout; may be null
    int64_t r_delta;           // byte distance R - Y: residual of *y is at y + r_delta
    int act;                   // olc_activation
};

// One launch's worth of work: `items` independent products
// [M, K] @ [K, N] -> [M, N] with operand offsets from `map`.  With a_trans
// A is stored [K, M] (row-major), with b_trans B is stored [N, K] (Gemm's
// transA / transB; rank-2 products only).
struct Problem {
    const void* A;
    const void* B;
    void* Y;
    int64_t M, N, K;
    int64_t items;
    BatchMap map;
    int split_hint;   // > 0: K slices requested by a tuning override, 0: automatic
    int variant;      // kernel-family override (0: automatic; see olc_matmul_plan_set_tc_variant)
    int a_trans, b_trans;
    Epilogue epi;
    // Row pitches in elements of A and B as the general tensor-core kernels
    // read them (0: dense, K for A and N for B).  A pitch above the row
    // length is a staged copy whose rows were padded to 16-byte multiples.
    int64_t a_ld, b_ld;
    // Y (or the residual) is not 16-byte aligned or N is not a multiple of
    // 8: the general tensor-core kernels store with 2-, 4- and 16-byte
    // accesses as each row's alignment allows.
    int y_unaligned;
    // General FP16/BF16 tiles: K slices per tile of the cluster split-K (0:
    // chosen from this problem's shape; 1: none; k >= 2: k).  Row chunks of
    // a larger product carry the whole product's choice, so that every
    // output element is summed in the same order as without chunks.
    int tc_ways;
};

// Workspace handed to the split reductions: `partials` holds fp32/fp64
// partial results, `counters` one arrival counter per output tile (zero
// between launches; the last arriving block resets its counter).
struct Workspace {
    void* partials;
    size_t partial_bytes;
    unsigned int* counters;
    size_t counter_count;
};

// Device error word (bounded waits that ran out set it).  Defined in
// simt.cu; device_error_word() is its device address on the current device.
cudaError_t read_and_clear_device_error(unsigned int* value, cudaStream_t stream);
unsigned int* device_error_word();

// ---- launchers: every one returns the launch's cudaError_t -------------

cudaError_t launch_zero_fill(void* Y, int64_t bytes, cudaStream_t stream);
// K == 0 with a Gemm epilogue: Y = beta * C (the product term is empty)
cudaError_t launch_epilogue_fill(olc_dtype dt, const Problem& p, cudaStream_t stream);

// DIRECT: small tiles, scalar loads, any shape and alignment.  FLOAT /
// DOUBLE products with K <= 256 / 128 (operands as given) fetch the whole K
// range of a tile at once (direct_wholek_ok).
cudaError_t launch_direct(olc_dtype dt, const Problem& p, cudaStream_t stream);
bool direct_wholek_ok(olc_dtype dt, const Problem& p);

// GENERAL_SIMT: FP32 FFMA / FP64 DFMA register-tiled kernel (any dtype works;
// the plan routes FLOAT and DOUBLE here).  FLOAT products with fewer tiles
// than SMs take `splits` > 1 K slices per tile (partial tiles in the
// workspace, summed in slice order by the last slice to finish).
cudaError_t launch_general_simt(olc_dtype dt, const Problem& p, cudaStream_t stream, int splits = 1,
                                const Workspace* ws = nullptr);
int general_simt_pick_split(olc_dtype dt, const Problem& p, int sm_count);
size_t general_simt_partial_bytes(olc_dtype dt, const Problem& p, int splits);
size_t general_simt_counter_count(olc_dtype dt, const Problem& p, int splits);
bool general_simt_vectorizable(olc_dtype dt, int64_t N, int64_t K);

// SKINNY_M: M <= 16.  `ksplit` slices of K, reduced in fixed order.
int skinny_m_max_rows();
cudaError_t launch_skinny_m(olc_dtype dt, const Problem& p, int ksplit, int sm_count,
                            const Workspace& ws, cudaStream_t stream, const void* bt_ready = nullptr);
size_t skinny_m_partial_bytes(olc_dtype dt, const Problem& p, int ksplit, int sm_count);
size_t skinny_m_counter_count(olc_dtype dt, const Problem& p, int ksplit, int sm_count);
int skinny_m_pick_split(olc_dtype dt, const Problem& p, int sm_count);

// SKINNY_M for E4M3FN / E5M2 on the tensor cores (fp8.cu): swapped operands,
// B transposed in shared memory on the way, K slices summed in slice order
bool f8_skinny_tc_ok(olc_dtype dt, const Problem& p);
int f8_skinny_tc_pick(const Problem& p, int sm_count);
size_t f8_skinny_tc_partial_bytes(const Problem& p, int ksplit);
size_t f8_skinny_tc_counter_count(const Problem& p, int ksplit);
// bt_ready: B already transposed ([N, K] bytes, a plan's constant B): the
// tiles go to the MMA as loaded, without the shared-memory transposition
cudaError_t launch_f8_skinny_tc(olc_dtype dt, const Problem& p, int ksplit, int sm_count, const Workspace& ws,
                                cudaStream_t stream, const void* bt_ready = nullptr);

// SKINNY_N: N <= 16.
int skinny_n_max_cols();
// E4M3FN / E5M2 products the register-streaming warp-MMA kernel takes (one
// B, K a multiple of 16, B within its shared-memory budget)
bool skinny_n_f8_ok(olc_dtype dt, const Problem& p);
cudaError_t launch_skinny_n(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                            cudaStream_t stream);
size_t skinny_n_partial_bytes(olc_dtype dt, const Problem& p, int sm_count);
size_t skinny_n_counter_count(olc_dtype dt, const Problem& p, int sm_count);

// SPLIT_K: tiny output, long K.  Partials in fixed-order reduction.  FLOAT16 /
// BFLOAT16 shapes with 16-byte row strides run on the tensor cores, the rest
// on the SIMT kernel.
cudaError_t launch_split_k(olc_dtype dt, const Problem& p, int splits, int sm_count,
                           const Workspace& ws, cudaStream_t stream);
size_t split_k_partial_bytes(olc_dtype dt, const Problem& p, int splits, int sm_count);
size_t split_k_counter_count(olc_dtype dt, const Problem& p, int splits, int sm_count);
int split_k_pick(olc_dtype dt, const Problem& p, int sm_count);
// the SIMT split-K kernel alone (32 x 32 tiles, one partial per slice)
cudaError_t launch_split_k_simt(olc_dtype dt, const Problem& p, int splits, const Workspace& ws,
                                cudaStream_t stream);
int split_k_simt_pick(olc_dtype dt, const Problem& p, int sm_count);

// SPLIT_K for E4M3FN / E5M2 with at most 32 rows and 128 columns (N a
// multiple of 16): warp-level MMA over K slices, two fixed-order levels.
bool f8_split_k_ok(olc_dtype dt, const Problem& p);
int f8_split_k_pick(const Problem& p, int sm_count);
size_t f8_split_k_partial_bytes(const Problem& p, int splits);
size_t f8_split_k_counter_count(const Problem& p, int splits);
cudaError_t launch_f8_split_k(olc_dtype dt, const Problem& p, int splits, const Workspace& ws,
                              cudaStream_t stream);

// 8-bit float operands (FLOAT output): SIMT decode kernel for any shape and
// batch; tcgen05 kind::f8f6f4 kernel for one item with K % 16 == 0 and
// N % 4 == 0 (B transposed into the workspace first)
cudaError_t launch_fp8_simt(olc_dtype dt, const Problem& p, cudaStream_t stream);
bool fp8_tc_ok(const Problem& p);
size_t fp8_tc_workspace_bytes(const Problem& p);
// bt_ready: B already transposed ([N, K] bytes; a plan's constant B), else
// the transpose runs into the workspace first
cudaError_t launch_fp8_tc(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                          cudaStream_t stream, const void* bt_ready = nullptr);
// B [K, N] bytes -> bt [N, K] bytes
cudaError_t launch_fp8_transpose(const Problem& p, void* bt, cudaStream_t stream);
// the CTA-pair tensor-core kernel on 8-bit float operands: A [M, K] and the
// transposed B [N, K] (bytes), float32 Y; one item, M and N >= 256
cudaError_t launch_pair_f8(olc_dtype dt, const Problem& p, const void* bt, int sm_count,
                           cudaStream_t stream);

// GENERAL_TC: tcgen05 tensor-core GEMM for FLOAT16 / BFLOAT16.
// tc_shape_ok: the dense operands are TMA-readable as given (16-byte rows).
bool tc_shape_ok(olc_dtype dt, int64_t N, int64_t K);
// cluster split-K slices the general FP16/BF16 tiles would use for this
// problem (0: none)
int tc_general_csplit_ways(olc_dtype dt, const Problem& p, int sm_count);
// Copy `rows` rows of `cols` 16-bit elements (src rows dense, any 2-byte
// alignment) into dst rows `pitch` elements apart (dst 16-byte aligned,
// pitch a multiple of 8 >= cols); the pitch's extra elements are zeroed.
cudaError_t launch_pad_rows16(const void* src, void* dst, int64_t rows, int64_t cols,
                              int64_t pitch, cudaStream_t stream);
// variant: 0 automatic, 1 one CTA per 128 x 256 tile, 2 CTA pairs (cta_group::2)
// with 256 x 256 tiles.  `ws` (may be null) holds the cluster split-K's
// partial tiles (tc_general_partial_bytes); without it those products run
// the plain tiles.
cudaError_t launch_general_tc(olc_dtype dt, const Problem& p, int sm_count, cudaStream_t stream,
                              int variant, const Workspace* ws);
// workspace of the cluster split-K for this problem (0: it does not apply)
size_t tc_general_partial_bytes(olc_dtype dt, const Problem& p, int sm_count);
// the same kernel with 16-column tiles (N <= 16): the tensor-core skinny-N,
// in stream-K shares when the row tiles alone leave SMs idle
size_t tc_skinny_n_partial_bytes(const Problem& p, int sm_count);
size_t tc_skinny_n_counter_count(const Problem& p, int sm_count);
cudaError_t launch_skinny_n_tc(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                               cudaStream_t stream);
// the same kernel in split-K mode (K slices per tile, two-level fixed-order
// reduction of float32 partial tiles)
int tc_split_pick(const Problem& p, int sm_count);
size_t tc_split_partial_bytes(const Problem& p, int sm_count);
size_t tc_split_counter_count(const Problem& p, int sm_count);
cudaError_t launch_tc_split(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                            cudaStream_t stream);
// the same kernel with swapped operands for M <= 16 (Y^T = B^T A^T): the
// tensor-core skinny-M, split over K when that fills the SMs better
int tc_skinny_m_pick(const Problem& p, int sm_count);
size_t tc_skinny_m_partial_bytes(const Problem& p, int sm_count);
size_t tc_skinny_m_counter_count(const Problem& p, int sm_count);
cudaError_t launch_tc_skinny_m(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                               cudaStream_t stream);

}  // namespace olc
