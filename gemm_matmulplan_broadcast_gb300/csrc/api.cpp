// Host side of the library: MatMulPlan (shape resolution, broadcast batch
// strides, batch collapse and folding), GemmPlan (algorithm choice, splits,
// workspace) and the exported C ABI.
//
// "MatMul Kernel Design", section "Shape and plan model": the plan resolves
// the whole output shape up front -- promoted M, N, K, the broadcast batch
// shape, per-operand batch strides with zeros for broadcast dimensions -- and
// embeds the GEMM plan that runs once per broadcast batch item.
// "Gemm and MatMul Performance Roadmap", section "Phase 4: complete MatMul":
// normalise rank-one inputs, compute zero-stride broadcast strides, collapse
// contiguous batch dimensions, dispatch the batches through the same
// scheduler, pick dedicated kernels for small M or N, and restore the output
// rank without copying.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "olc_internal.h"

using namespace olc;

struct olc_matmul_plan {
    olc_dtype dtype;
    int a_rank, b_rank;
    int64_t a_shape[OLC_MAX_RANK], b_shape[OLC_MAX_RANK];
    // resolved shape
    int out_rank;
    int64_t out_shape[OLC_MAX_RANK];
    int64_t M, N, K;
    int64_t batch;               // number of broadcast batch items
    int batch_rank;
    int64_t batch_shape[OLC_MAX_RANK];
    int64_t a_bstride[OLC_MAX_RANK], b_bstride[OLC_MAX_RANK];
    // launch geometry after collapse / fold
    int64_t rows;                // M times the folded batch
    int64_t items;               // batch items a launch walks
    BatchMap map;
    // GEMM plan
    int algo;
    bool forced;
    int splits;                  // SPLIT_K slices or SKINNY_M K-slices
    int split_hint;              // tuning override of the slice count (0 = automatic)
    int tc_variant;              // tuning override of the tensor-core tiling (0 = automatic)
    int cluster_slices;          // GENERAL_TC FLOAT16 / BFLOAT16: K slices of the cluster split-K (1: none)
    // Gemm operator (rank-2, transA / transB, alpha, beta, broadcast C)
    int is_gemm;
    int trans_a, trans_b;
    double alpha, beta;
    int c_rank;                  // -1: no C
    int64_t c_shape[2];
    int64_t c_rs, c_cs;          // element strides of C over [M, N] (0 = broadcast)
    // plan-owned constant B (device copy on the plan's device)
    void* const_b;
    size_t const_b_bytes;
    int const_b_set;
    void* const_bt;              // 8-bit float tensor-core plans: constant B as [N, K] bytes
    size_t const_bt_bytes;
    int f8_const_tc;             // 8-bit few-row plan moved to the tcgen05 kernel by its constant B
    void* const_b_pad;           // 16-bit plans with N % 8 != 0: constant B, rows padded to 16 bytes
    size_t const_b_pad_bytes;
    // staging copies of operands the tensor-core kernels cannot read in
    // place (rows not a multiple of 16 bytes, or a pointer off a 16-byte
    // boundary): A's copy, then B's, 256-byte aligned
    void* stage;
    size_t stage_bytes;
    // fused epilogue: activation, and a residual in the output's layout
    int act;
    int residual;
    // host-buffer pipeline: copy streams and per-chunk events (created at
    // the first pipelined olc_matmul_execute_host)
    cudaStream_t copy_in, copy_out;
    cudaEvent_t ev_start, ev_b, ev_done;
    cudaEvent_t ev_a[8], ev_y[8];
    int pipe_ready;
    int device;                  // -1: planned without a device
    int sm_count;
    void* workspace;
    size_t ws_bytes;
    size_t partial_bytes;
    size_t counter_count;
    // the last execute that used the workspace or the staging buffer:
    // an execute on another stream waits for it (created at first use)
    cudaEvent_t state_ev;
    cudaStream_t state_stream;
    int state_ev_live;           // state_ev marks the last such execute
    // row chunks of a host-buffer pipeline: the whole product's cluster
    // split-K choice (0 on every plan; set on the chunk copies only)
    int chunk_tc_ways;
};

namespace {

constexpr int kDefaultSmCount = 152;   // GB300; used only when no device is visible

// bytes of one operand element
int64_t elem_bytes(olc_dtype dt) {
    switch (dt) {
        case OLC_FLOAT: return 4;
        case OLC_DOUBLE: return 8;
        case OLC_FLOAT16:
        case OLC_BFLOAT16: return 2;
        case OLC_FLOAT8E4M3FN:
        case OLC_FLOAT8E4M3FNUZ:
        case OLC_FLOAT8E5M2:
        case OLC_FLOAT8E5M2FNUZ: return 1;
    }
    return 0;
}

bool valid_dtype(int dt) {
    return dt == OLC_FLOAT || dt == OLC_DOUBLE || dt == OLC_FLOAT16 || dt == OLC_BFLOAT16 ||
           dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2 || dt == OLC_FLOAT8E4M3FNUZ ||
           dt == OLC_FLOAT8E5M2FNUZ;
}

bool is_half(olc_dtype dt) { return dt == OLC_FLOAT16 || dt == OLC_BFLOAT16; }
bool is_fp8(olc_dtype dt) {
    return dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2 || dt == OLC_FLOAT8E4M3FNUZ ||
           dt == OLC_FLOAT8E5M2FNUZ;
}
// the 8-bit formats the tensor cores take (kind::f8f6f4 E4M3 / E5M2)
bool is_fp8_tc_format(olc_dtype dt) { return dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2; }

// bytes of one output element: FLOAT for the 8-bit float operand types
int64_t out_bytes(olc_dtype dt) { return is_fp8(dt) ? 4 : elem_bytes(dt); }

int64_t out_numel(const olc_matmul_plan* p) {
    int64_t n = 1;
    for (int i = 0; i < p->out_rank; ++i) n *= p->out_shape[i];
    return n;
}

int64_t numel(const int64_t* s, int r) {
    int64_t n = 1;
    for (int i = 0; i < r; ++i) n *= s[i];
    return n;
}

// Largest tensor the plans accept, in bytes: 2^62, so that every element and
// byte offset the kernels form (and sums of two of them) fits in int64.
constexpr int64_t kMaxTensorBytes = int64_t(1) << 62;

// true when the tensor of these extents, `elem` bytes per element, stays
// within kMaxTensorBytes (an extent of 0 makes it empty, which always fits)
bool tensor_fits(const int64_t* s, int r, int64_t elem) {
    for (int i = 0; i < r; ++i)
        if (s[i] == 0) return true;
    int64_t n = elem;
    for (int i = 0; i < r; ++i)
        if (__builtin_mul_overflow(n, s[i], &n) || n > kMaxTensorBytes) return false;
    return true;
}

Problem make_problem(const olc_matmul_plan* p, const void* A, const void* B, void* Y,
                     const void* C = nullptr, const void* R = nullptr) {
    Problem pr;
    std::memset(&pr, 0, sizeof pr);
    pr.A = A;
    pr.B = B;
    pr.Y = Y;
    pr.M = p->rows;
    pr.N = p->N;
    pr.K = p->K;
    pr.items = p->items;
    pr.map = p->map;
    pr.split_hint = p->split_hint;
    // an 8-bit few-row plan with a constant B runs the tcgen05 kernel
    // (variant 3) unless a kernel family was asked for
    pr.variant = (p->f8_const_tc && (p->tc_variant == 0 || p->tc_variant == 3)) ? 3 : p->tc_variant;
    pr.tc_ways = p->chunk_tc_ways;
    pr.a_trans = p->trans_a;
    pr.b_trans = p->trans_b;
    // Gemm: alpha * acc + beta * C, then the fused residual and activation;
    // the plain product when alpha is 1 and nothing else is asked for (the
    // same results, without the epilogue's work)
    const bool gemm_epi = p->is_gemm && (p->alpha != 1.0 || p->c_rank >= 0);
    if (gemm_epi || p->act != OLC_ACT_NONE || p->residual) {
        const double alpha = p->is_gemm ? p->alpha : 1.0;
        const double beta = p->is_gemm ? p->beta : 0.0;
        pr.epi.mode = 1;
        pr.epi.alpha_f = (float)alpha;
        pr.epi.beta_f = (float)beta;
        pr.epi.alpha_d = alpha;
        pr.epi.beta_d = beta;
        pr.epi.C = p->is_gemm && p->c_rank >= 0 ? C : nullptr;
        pr.epi.c_rs = p->c_rs;
        pr.epi.c_cs = p->c_cs;
        pr.epi.R = p->residual ? R : nullptr;
        pr.epi.r_delta = p->residual ? (int64_t)(reinterpret_cast<intptr_t>(R) -
                                                 reinterpret_cast<intptr_t>(Y))
                                     : 0;
        pr.epi.act = p->act;
    }
    return pr;
}

// Collapse the broadcast batch dimensions: drop extent-1 dimensions, then
// merge neighbours whose strides chain for both operands (the output is dense,
// so its strides always chain).  Then fold: when B is shared by every item
// and A's items are consecutive matrices, the items become extra rows of one
// GEMM (M' = items * M).
void collapse_and_fold(olc_matmul_plan* p) {
    BatchMap m;
    std::memset(&m, 0, sizeof m);
    for (int d = 0; d < p->batch_rank; ++d) {
        if (p->batch_shape[d] == 1) continue;
        const int64_t e = p->batch_shape[d];
        const int64_t sa = p->a_bstride[d], sb = p->b_bstride[d];
        if (m.rank > 0) {
            const int q = m.rank - 1;
            if (m.a_stride[q] == sa * e && m.b_stride[q] == sb * e) {
                m.dims[q] *= e;
                m.a_stride[q] = sa;
                m.b_stride[q] = sb;
                continue;
            }
        }
        m.dims[m.rank] = e;
        m.a_stride[m.rank] = sa;
        m.b_stride[m.rank] = sb;
        ++m.rank;
    }
    p->rows = p->M;
    p->items = p->batch;
    if (m.rank == 1 && m.b_stride[0] == 0 && m.a_stride[0] == p->M * p->K) {
        p->rows = p->M * m.dims[0];
        p->items = 1;
        m.rank = 0;
    }
    p->map = m;
}

// Shapes each algorithm can take (dtype, N, K; pointer alignment is checked
// at execute time).
bool feasible(const olc_matmul_plan* p, int algo) {
    const int64_t rows = p->rows, N = p->N, K = p->K;
    const int64_t n = out_numel(p);
    if (is_fp8(p->dtype)) {
        switch (algo) {
            case OLC_ALGO_EMPTY: return n == 0;
            case OLC_ALGO_ZERO_FILL: return n > 0 && K == 0;
            case OLC_ALGO_DIRECT:
            case OLC_ALGO_GENERAL_SIMT: return n > 0 && K > 0;
            case OLC_ALGO_SKINNY_M:     // 16 one-byte B elements per vector
                return n > 0 && K > 0 && rows <= skinny_m_max_rows() && N % 16 == 0;
            case OLC_ALGO_SPLIT_K: {    // warp-MMA split-K: small outputs
                Problem pr = make_problem(p, nullptr, nullptr, nullptr);
                return n > 0 && f8_split_k_ok(p->dtype, pr);
            }
            case OLC_ALGO_SKINNY_N: {   // warp-MMA streaming of A: N <= 16
                Problem pr = make_problem(p, nullptr, nullptr, nullptr);
                return n > 0 && K > 0 && skinny_n_f8_ok(p->dtype, pr);
            }
            case OLC_ALGO_GENERAL_TC: {
                Problem pr = make_problem(p, nullptr, nullptr, nullptr);
                return n > 0 && K > 0 && is_fp8_tc_format(p->dtype) && fp8_tc_ok(pr);
            }
        }
        return false;
    }
    const bool trans = p->trans_a || p->trans_b;
    if (trans && (algo == OLC_ALGO_SKINNY_M || algo == OLC_ALGO_SKINNY_N || algo == OLC_ALGO_SPLIT_K))
        return false;   // transposed operands: general and direct kernels only
    if (algo == OLC_ALGO_GENERAL_TC && p->trans_a && (p->M * elem_bytes(p->dtype)) % 16 != 0)
        return false;   // A stored [K, M] needs 16-byte rows for TMA
    switch (algo) {
        case OLC_ALGO_EMPTY: return n == 0;
        case OLC_ALGO_ZERO_FILL: return n > 0 && K == 0;
        case OLC_ALGO_DIRECT:
        case OLC_ALGO_GENERAL_SIMT: return n > 0 && K > 0;
        case OLC_ALGO_SKINNY_M:
            return n > 0 && K > 0 && rows <= skinny_m_max_rows() &&
                   (N * elem_bytes(p->dtype)) % 16 == 0;
        case OLC_ALGO_SKINNY_N:
            return n > 0 && K > 0 && N <= skinny_n_max_cols() &&
                   (K * elem_bytes(p->dtype)) % 16 == 0;
        case OLC_ALGO_SPLIT_K:
            return n > 0 && K > 0 && (K * elem_bytes(p->dtype)) % 16 == 0 &&
                   (N * elem_bytes(p->dtype)) % 16 == 0;
        case OLC_ALGO_GENERAL_TC:
            // operands whose rows are not 16-byte multiples are staged into
            // padded rows first (A as [M, K], B as [K, N]); transposed
            // operands are read in place and need 16-byte rows
            return n > 0 && K > 0 && is_half(p->dtype) && rows < (1LL << 31) && N < (1LL << 31) &&
                   K < (1LL << 31) && (!p->trans_b || K % 8 == 0);
    }
    return false;
}

// ---- staging copies for the tensor-core kernels --------------------------

// An operand as stored: `rows` rows of `cols` 16-bit elements.
struct StoredRows {
    int64_t rows, cols;
};
StoredRows stored_a(const olc_matmul_plan* p) {
    const int64_t cols = p->trans_a ? p->M : p->K;
    const int64_t total = numel(p->a_shape, p->a_rank);
    return {cols > 0 ? total / cols : 0, cols};
}
StoredRows stored_b(const olc_matmul_plan* p) {
    const int64_t cols = p->trans_b ? p->K : p->N;
    const int64_t total = numel(p->b_shape, p->b_rank);
    return {cols > 0 ? total / cols : 0, cols};
}
int64_t pad8(int64_t n) { return (n + 7) / 8 * 8; }
size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Staging copies an execute needs (16-bit plans on the tensor-core, skinny
// and split-K kernels, which read A and B with TMA or 16-byte vectors).  An
// operand is copied when its pointer is off a 16-byte boundary or, for the
// general tensor-core tiles (`tc`), when its stored rows are not a multiple
// of 16 bytes.  The general tiles take the copy with rows padded to 8
// elements (read through a row pitch); the other kernels take a dense copy.
struct StageNeed {
    bool a, b;
    size_t a_bytes, b_bytes;
};
StageNeed stage_need(const olc_matmul_plan* p, const void* A, const void* B, bool tc,
                     bool b_padded) {
    StageNeed n{false, false, 0, 0};
    const StoredRows ra = stored_a(p), rb = stored_b(p);
    n.a = (reinterpret_cast<uintptr_t>(A) & 15) != 0 || (tc && ra.cols % 8 != 0);
    n.b = !b_padded && ((reinterpret_cast<uintptr_t>(B) & 15) != 0 || (tc && rb.cols % 8 != 0));
    auto bytes = [&](const StoredRows& r) {
        return round256((size_t)(tc ? r.rows * pad8(r.cols) : pad8(r.rows * r.cols)) * 2);
    };
    if (n.a) n.a_bytes = bytes(ra);
    if (n.b) n.b_bytes = bytes(rb);
    return n;
}

void free_stage(olc_matmul_plan* p) {
    if (p->stage) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (p->device >= 0 && cur != p->device) cudaSetDevice(p->device);
        cudaFree(p->stage);
        if (p->device >= 0 && cur >= 0 && cur != p->device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    p->stage = nullptr;
    p->stage_bytes = 0;
}

// Grow the staging buffer to `bytes` (cudaMalloc on the plan's device; the
// previous buffer is freed first, which waits for work using it).
olc_status ensure_stage(olc_matmul_plan* p, size_t bytes) {
    if (bytes <= p->stage_bytes) return OLC_OK;
    free_stage(p);
    void* mem = nullptr;
    if (cudaMalloc(&mem, bytes) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_OOM;
    }
    p->stage = mem;
    p->stage_bytes = bytes;
    return OLC_OK;
}

int choose_algorithm(const olc_matmul_plan* p) {
    if (out_numel(p) == 0) return OLC_ALGO_EMPTY;
    if (p->K == 0) return OLC_ALGO_ZERO_FILL;
    if (is_fp8(p->dtype)) {
        const double macs = (double)p->rows * (double)p->N * (double)p->K * (double)p->items;
        if (p->rows <= skinny_m_max_rows() && p->N >= 256 && feasible(p, OLC_ALGO_SKINNY_M))
            return OLC_ALGO_SKINNY_M;
        // few columns: the warp-MMA streaming kernel up to 8 columns (one
        // [16384, 4096] x [4096, 8] E4M3FN product: 22.0 us against 36.8 on
        // the tensor-core tile kernel); at 9-16 columns its four FP8 MMAs per
        // chunk make it no faster than the tile kernel (33.3 against 32.2 us)
        if (p->N <= 8 && p->rows >= 256 && feasible(p, OLC_ALGO_SKINNY_N))
            return OLC_ALGO_SKINNY_N;
        // the split-K corner, as for the other types: too few output tiles to
        // fill half the SMs, and a long K
        const int64_t tiles = ((p->rows + 127) / 128) * ((p->N + 127) / 128) * p->items;
        if (tiles * 2 <= p->sm_count && p->K >= 8 * 1024 && feasible(p, OLC_ALGO_SPLIT_K))
            return OLC_ALGO_SPLIT_K;
        if (macs >= 4.0 * 1024 * 1024 && feasible(p, OLC_ALGO_GENERAL_TC)) return OLC_ALGO_GENERAL_TC;
        return macs < 4.0 * 1024 * 1024 ? OLC_ALGO_DIRECT : OLC_ALGO_GENERAL_SIMT;
    }
    const int64_t rows = p->rows, N = p->N, K = p->K, items = p->items;
    const double macs = (double)rows * (double)N * (double)K * (double)items;
    if (rows <= skinny_m_max_rows() && N >= 256 && feasible(p, OLC_ALGO_SKINNY_M))
        return OLC_ALGO_SKINNY_M;
    if (N <= skinny_n_max_cols() && rows >= 256 && feasible(p, OLC_ALGO_SKINNY_N))
        return OLC_ALGO_SKINNY_N;
    if (macs < 4.0 * 1024 * 1024) return OLC_ALGO_DIRECT;
    // Split-K only for the guarded corner: too few output tiles (counting the
    // batch, which takes priority) to fill half the SMs, and a long K.
    const int64_t tiles = ((rows + 127) / 128) * ((N + 127) / 128) * items;
    if (tiles * 2 <= p->sm_count && K >= 8 * 1024 && feasible(p, OLC_ALGO_SPLIT_K)) {
        // FLOAT16 / BFLOAT16 outputs above 32 x 32 whose general tiles take
        // the cluster split-K (slices summed from L2 in slice order within
        // one cluster) stay there: faster than the global two-level
        // reduction (BF16 [64, 8192] x [8192, 512]: 12.2 against 38.4 us;
        // [128, 16384] x [16384, 1024]: 20.1 against 71.8 us)
        const bool tiny_out = rows <= 32 && N <= 32 && items == 1;
        if (!(is_half(p->dtype) && !tiny_out && feasible(p, OLC_ALGO_GENERAL_TC) &&
              tc_general_csplit_ways(p->dtype, make_problem(p, nullptr, nullptr, nullptr), p->sm_count) >= 2))
            return OLC_ALGO_SPLIT_K;
    }
    // Short-K FLOAT / DOUBLE products that leave the register-tile kernel
    // few tiles per SM: DIRECT's whole-K 32 x 32 tiles (one global round
    // trip per tile, four times as many blocks) are faster.  Measured on
    // GB300 (us, whole-K against register tiles): FLOAT 512x256x512 14 / 26,
    // 1024x256x64 9 / 25, 256x256x2048 25 / 26, but 1024x256x1024 43 / 27;
    // DOUBLE 1024x128x1024 227 / 260, 2048x64x512 115 / 132.
    if (!is_half(p->dtype)) {
        const Problem pr = make_problem(p, nullptr, nullptr, nullptr);
        const int64_t tiles64 = ((rows + 63) / 64) * ((N + 63) / 64) * items;
        const bool few = p->dtype == OLC_FLOAT ? tiles * 4 <= p->sm_count : tiles64 <= 4 * p->sm_count;
        if (few && direct_wholek_ok(p->dtype, pr)) return OLC_ALGO_DIRECT;
    }
    if (is_half(p->dtype) && feasible(p, OLC_ALGO_GENERAL_TC)) return OLC_ALGO_GENERAL_TC;
    return is_half(p->dtype) ? OLC_ALGO_DIRECT : OLC_ALGO_GENERAL_SIMT;
}

void free_workspace(olc_matmul_plan* p) {
    if (p->workspace) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (p->device >= 0 && cur != p->device) cudaSetDevice(p->device);
        cudaFree(p->workspace);
        if (p->device >= 0 && cur >= 0 && cur != p->device) cudaSetDevice(cur);
    }
    p->workspace = nullptr;
    p->ws_bytes = 0;
    p->partial_bytes = 0;
    p->counter_count = 0;
}

// Size (and, with a device, allocate) the workspace for the current choice.
olc_status prepare_algorithm(olc_matmul_plan* p) {
    free_workspace(p);
    p->splits = 1;
    p->cluster_slices = 1;
    Problem pr = make_problem(p, nullptr, nullptr, nullptr);
    const olc_dtype dt = p->dtype;
    if (p->algo == OLC_ALGO_SPLIT_K) {
        p->splits = split_k_pick(dt, pr, p->sm_count);
        p->partial_bytes = split_k_partial_bytes(dt, pr, p->splits, p->sm_count);
        p->counter_count = split_k_counter_count(dt, pr, p->splits, p->sm_count);
    } else if (p->algo == OLC_ALGO_SKINNY_N) {
        p->partial_bytes = skinny_n_partial_bytes(dt, pr, p->sm_count);
        p->counter_count = skinny_n_counter_count(dt, pr, p->sm_count);
    } else if (p->algo == OLC_ALGO_GENERAL_TC && is_fp8(dt)) {
        p->partial_bytes = fp8_tc_workspace_bytes(pr);    // B transposed, [N, K] bytes
    } else if (p->algo == OLC_ALGO_GENERAL_TC && is_half(dt) && p->tc_variant == 0) {
        // few tiles: the cluster split-K's float32 partial tiles
        p->partial_bytes = tc_general_partial_bytes(dt, pr, p->sm_count);
        if (p->partial_bytes > 0) p->cluster_slices = tc_general_csplit_ways(dt, pr, p->sm_count);
    } else if (p->algo == OLC_ALGO_GENERAL_SIMT) {
        p->splits = general_simt_pick_split(dt, pr, p->sm_count);
        if (p->splits > 1) {
            p->partial_bytes = general_simt_partial_bytes(dt, pr, p->splits);
            p->counter_count = general_simt_counter_count(dt, pr, p->splits);
        }
    } else if (p->algo == OLC_ALGO_SKINNY_M) {
        p->splits = skinny_m_pick_split(dt, pr, p->sm_count);
        if (p->splits > 1) {
            p->partial_bytes = skinny_m_partial_bytes(dt, pr, p->splits, p->sm_count);
            p->counter_count = skinny_m_counter_count(dt, pr, p->splits, p->sm_count);
        }
    }
    // 16-bit tensor-core plans whose operand rows are not 16-byte multiples
    // stage those operands at every execute: the copy buffer belongs to the
    // plan from here on (pointer misalignment alone is only known at execute)
    if (p->algo == OLC_ALGO_GENERAL_TC && is_half(dt) && p->device >= 0) {
        const StageNeed need = stage_need(p, nullptr, nullptr, true, p->const_b_pad != nullptr);
        if (need.a_bytes + need.b_bytes > 0) {
            const olc_status st = ensure_stage(p, need.a_bytes + need.b_bytes);
            if (st != OLC_OK) return st;
        }
    }
    if (p->partial_bytes == 0 && p->counter_count == 0) return OLC_OK;
    const size_t counters_off = (p->partial_bytes + 255) / 256 * 256;
    p->ws_bytes = counters_off + p->counter_count * sizeof(unsigned int);
    if (p->device < 0) return OLC_OK;   // allocated at the first execute
    void* ws = nullptr;
    if (cudaMalloc(&ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        p->ws_bytes = 0;
        return OLC_ERR_OOM;
    }
    if (cudaMemset(ws, 0, p->ws_bytes) != cudaSuccess) {
        cudaFree(ws);
        p->ws_bytes = 0;
        return OLC_ERR_CUDA;
    }
    p->workspace = ws;
    return OLC_OK;
}

Workspace workspace_of(const olc_matmul_plan* p) {
    Workspace w;
    const size_t counters_off = (p->partial_bytes + 255) / 256 * 256;
    w.partials = p->workspace;
    w.partial_bytes = p->partial_bytes;
    w.counters = p->workspace ? reinterpret_cast<unsigned int*>(
                                    static_cast<char*>(p->workspace) + counters_off)
                              : nullptr;
    w.counter_count = p->counter_count;
    return w;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

olc_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return OLC_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? OLC_ERR_OOM : OLC_ERR_CUDA;
}

// The kernels an execute with these pointers runs.  FLOAT16 / BFLOAT16 stay
// on the tensor cores whatever the alignment: operands the kernels cannot
// read in place are copied first (stage_need), and the general kernels store
// a Y of any alignment; the skinny and split-K kernels store with 16-byte
// vectors, so a misaligned Y (or residual) moves their products to the
// general kernels.  Other types: a misaligned pointer sends the product to
// the DIRECT kernel.
struct Route {
    int algo;
    bool tc;            // general tensor-core tiles
    bool b_padded;      // B is the plan's constant B, already in padded rows
    bool y_unaligned;   // Y stored by alignment
    StageNeed need;
};
Route route_of(const olc_matmul_plan* p, const void* A, const void* B, const void* Y, const void* R) {
    Route r;
    r.algo = p->algo;
    r.tc = false;
    r.b_padded = false;
    r.y_unaligned = false;
    r.need = StageNeed{false, false, 0, 0};
    const int a = p->algo;
    if (a == OLC_ALGO_EMPTY || a == OLC_ALGO_ZERO_FILL || a == OLC_ALGO_DIRECT ||
        a == OLC_ALGO_GENERAL_SIMT)
        return r;
    if (is_half(p->dtype)) {
        const bool yr_off = !aligned16(Y) || (R && !aligned16(R));
        if (yr_off && a != OLC_ALGO_GENERAL_TC)
            r.algo = feasible(p, OLC_ALGO_GENERAL_TC) ? OLC_ALGO_GENERAL_TC : OLC_ALGO_DIRECT;
        if (r.algo == OLC_ALGO_DIRECT) return r;
        r.tc = r.algo == OLC_ALGO_GENERAL_TC;
        r.b_padded = r.tc && p->const_b_pad && B == p->const_b;
        r.need = stage_need(p, A, B, r.tc, r.b_padded);
        r.y_unaligned = r.tc && (yr_off || p->N % 8 != 0);
        return r;
    }
    // the residual is read with the same vector widths as Y is written
    const bool al = aligned16(A) && aligned16(B) && aligned16(Y) && (!R || aligned16(R));
    if (!al) r.algo = OLC_ALGO_DIRECT;
    return r;
}

cudaError_t launch_route(const olc_matmul_plan* p, const Problem& pr, olc_dtype dt, int algo,
                         const void* B, cudaStream_t s);

// Executes that use the plan's workspace (split partials and counters, the
// per-call FP8 transpose of B) or its staging buffer must not overlap on
// the GPU.  An execute on another stream than the last such one waits for
// it (cudaStreamWaitEvent), so calls from several streams are serialised
// on that state instead of racing; on one stream, stream order does it.
// Nothing is recorded or waited for while `s` is capturing a graph:
// ordering captured work is the graph's.
cudaError_t order_after_state_use(olc_matmul_plan* p, cudaStream_t s) {
    if (!p->state_ev_live || p->state_stream == s) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;
    return cudaStreamWaitEvent(s, p->state_ev, 0);
}

cudaError_t note_state_use(olc_matmul_plan* p, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) {
        p->state_ev_live = 0;        // a captured use is ordered by its graph
        return cudaSuccess;
    }
    if (!p->state_ev) {
        e = cudaEventCreateWithFlags(&p->state_ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    e = cudaEventRecord(p->state_ev, s);
    if (e != cudaSuccess) return e;
    p->state_stream = s;
    p->state_ev_live = 1;
    return cudaSuccess;
}

olc_status run(const olc_matmul_plan* p, const void* A, const void* B, void* Y, cudaStream_t s,
               const void* C = nullptr, const void* R = nullptr) {
    const int64_t n = out_numel(p);
    if (p->algo == OLC_ALGO_EMPTY || n == 0) return OLC_OK;
    if (!Y) return OLC_ERR_NULL;
    if (p->is_gemm && p->c_rank >= 0 && !C) return OLC_ERR_NULL;
    if (p->residual && !R) return OLC_ERR_NEEDS_RESIDUAL;
    if (p->algo == OLC_ALGO_ZERO_FILL) {
        Problem zp = make_problem(p, A, B, Y, C, R);
        if (zp.epi.mode) return from_cuda(launch_epilogue_fill(p->dtype, zp, s));
        return from_cuda(launch_zero_fill(Y, n * out_bytes(p->dtype), s));
    }
    if (!A || !B) return OLC_ERR_NULL;
    // every pointer must be aligned to its element size (the kernels load
    // and store whole elements)
    {
        const uintptr_t ein = (uintptr_t)elem_bytes(p->dtype) - 1, eout = (uintptr_t)out_bytes(p->dtype) - 1;
        if ((reinterpret_cast<uintptr_t>(A) & ein) || (reinterpret_cast<uintptr_t>(B) & ein) ||
            (reinterpret_cast<uintptr_t>(Y) & eout) || (reinterpret_cast<uintptr_t>(C) & ein) ||
            (reinterpret_cast<uintptr_t>(R) & eout))
            return OLC_ERR_INVALID;
    }
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return from_cuda(cudaErrorNoDevice);
    if (p->device >= 0 && cur != p->device) return OLC_ERR_WRONG_DEVICE;
    olc_matmul_plan* mp = const_cast<olc_matmul_plan*>(p);
    if (p->device < 0) {
        // planned on a machine view without a device: bind now
        mp->device = cur;
        if ((p->partial_bytes > 0 || p->counter_count > 0) && !p->workspace) {
            olc_status st = prepare_algorithm(mp);
            if (st != OLC_OK) return st;
        }
    }
    Problem pr = make_problem(p, A, B, Y, C, R);
    const olc_dtype dt = p->dtype;
    const Route rt = route_of(p, A, B, Y, R);
    const int algo = rt.algo;
    cudaError_t e = cudaSuccess;
    const bool uses_state = p->workspace != nullptr || rt.need.a || rt.need.b;
    if (uses_state) {
        e = order_after_state_use(mp, s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (rt.need.a || rt.need.b) {
        const olc_status st = ensure_stage(mp, rt.need.a_bytes + rt.need.b_bytes);
        if (st != OLC_OK) return st;
        unsigned char* base = static_cast<unsigned char*>(p->stage);
        // copy one operand: padded rows for the general tiles, one dense run
        // otherwise; `ld` receives the row pitch the kernels read (0: dense)
        auto stage = [&](const void* src, void* dst, const StoredRows& r, int64_t& ld) {
            if (rt.tc) {
                ld = pad8(r.cols) != r.cols ? pad8(r.cols) : 0;
                return launch_pad_rows16(src, dst, r.rows, r.cols, pad8(r.cols), s);
            }
            ld = 0;
            return launch_pad_rows16(src, dst, 1, r.rows * r.cols, pad8(r.rows * r.cols), s);
        };
        if (rt.need.a) {
            e = stage(A, base, stored_a(p), pr.a_ld);
            if (e != cudaSuccess) return from_cuda(e);
            pr.A = base;
        }
        if (rt.need.b) {
            e = stage(B, base + rt.need.a_bytes, stored_b(p), pr.b_ld);
            if (e != cudaSuccess) return from_cuda(e);
            pr.B = base + rt.need.a_bytes;
        }
    }
    if (rt.b_padded) {
        pr.B = p->const_b_pad;
        pr.b_ld = pad8(stored_b(p).cols);
    }
    pr.y_unaligned = rt.y_unaligned ? 1 : 0;
    if (algo < OLC_ALGO_DIRECT || algo > OLC_ALGO_GENERAL_SIMT) return OLC_ERR_INVALID;
    e = launch_route(p, pr, dt, algo, B, s);
    if (e == cudaSuccess && uses_state) e = note_state_use(mp, s);
    return from_cuda(e);
}

cudaError_t launch_route(const olc_matmul_plan* p, const Problem& pr, olc_dtype dt, int algo,
                         const void* B, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (is_fp8(dt)) {
        // the plan's constant B comes transposed already
        const void* bt = (p->const_bt && B == p->const_b) ? p->const_bt : nullptr;
        if (algo == OLC_ALGO_SKINNY_M)
            e = launch_skinny_m(dt, pr, p->splits, p->sm_count, workspace_of(p), s, bt);
        else if (algo == OLC_ALGO_SPLIT_K)
            e = launch_split_k(dt, pr, p->splits, p->sm_count, workspace_of(p), s);
        else if (algo == OLC_ALGO_SKINNY_N)
            e = launch_skinny_n(dt, pr, p->sm_count, workspace_of(p), s);
        else
            e = algo == OLC_ALGO_GENERAL_TC ? launch_fp8_tc(dt, pr, p->sm_count, workspace_of(p), s, bt)
                                            : launch_fp8_simt(dt, pr, s);
        return e;
    }
    switch (algo) {
        case OLC_ALGO_DIRECT: e = launch_direct(dt, pr, s); break;
        case OLC_ALGO_GENERAL_SIMT: {
            const Workspace ws = workspace_of(p);
            e = launch_general_simt(dt, pr, s, p->splits, &ws);
            break;
        }
        case OLC_ALGO_SKINNY_M:
            e = launch_skinny_m(dt, pr, p->splits, p->sm_count, workspace_of(p), s);
            break;
        case OLC_ALGO_SKINNY_N: e = launch_skinny_n(dt, pr, p->sm_count, workspace_of(p), s); break;
        case OLC_ALGO_SPLIT_K:
            e = launch_split_k(dt, pr, p->splits, p->sm_count, workspace_of(p), s);
            break;
        case OLC_ALGO_GENERAL_TC: {
            const Workspace ws = workspace_of(p);
            e = launch_general_tc(dt, pr, p->sm_count, s, p->tc_variant, &ws);
            break;
        }
        default: return cudaErrorInvalidValue;
    }
    return e;
}

}  // namespace

// ===========================================================================
// exported ABI

extern "C" {

olc_status olc_matmul_plan_create(const int64_t* a_shape, int a_rank, const int64_t* b_shape,
                                  int b_rank, olc_dtype dtype, olc_matmul_plan** out) {
    if (!out) return OLC_ERR_NULL;
    *out = nullptr;
    if ((!a_shape && a_rank > 0) || (!b_shape && b_rank > 0)) return OLC_ERR_NULL;
    if (a_rank < 1 || b_rank < 1 || a_rank > OLC_MAX_RANK || b_rank > OLC_MAX_RANK)
        return OLC_ERR_RANK;
    if (!valid_dtype(dtype)) return OLC_ERR_DTYPE;
    for (int i = 0; i < a_rank; ++i)
        if (a_shape[i] < 0) return OLC_ERR_NEGATIVE_DIM;
    for (int i = 0; i < b_rank; ++i)
        if (b_shape[i] < 0) return OLC_ERR_NEGATIVE_DIM;
    if (!tensor_fits(a_shape, a_rank, elem_bytes(dtype)) || !tensor_fits(b_shape, b_rank, elem_bytes(dtype)))
        return OLC_ERR_INVALID;

    olc_matmul_plan* p = new (std::nothrow) olc_matmul_plan;
    if (!p) return OLC_ERR_OOM;
    std::memset(p, 0, sizeof *p);
    p->dtype = dtype;
    p->a_rank = a_rank;
    p->b_rank = b_rank;
    std::memcpy(p->a_shape, a_shape, sizeof(int64_t) * a_rank);
    std::memcpy(p->b_shape, b_shape, sizeof(int64_t) * b_rank);
    p->device = -1;

    // 1. rank-one promotion: A [K] -> [1, K], B [K] -> [K, 1]
    int64_t a2[OLC_MAX_RANK + 1], b2[OLC_MAX_RANK + 1];
    int ra2 = a_rank, rb2 = b_rank;
    if (a_rank == 1) { a2[0] = 1; a2[1] = a_shape[0]; ra2 = 2; }
    else std::memcpy(a2, a_shape, sizeof(int64_t) * a_rank);
    if (b_rank == 1) { b2[0] = b_shape[0]; b2[1] = 1; rb2 = 2; }
    else std::memcpy(b2, b_shape, sizeof(int64_t) * b_rank);
    p->M = a2[ra2 - 2];
    p->K = a2[ra2 - 1];
    p->N = b2[rb2 - 1];
    if (b2[rb2 - 2] != p->K) { delete p; return OLC_ERR_K_MISMATCH; }

    // 2. multidirectional broadcast of the batch dimensions (right-aligned)
    const int ba = ra2 - 2, bb = rb2 - 2;
    const int r = std::max(ba, bb);
    // each operand's own contiguous batch strides
    int64_t a_own[OLC_MAX_RANK], b_own[OLC_MAX_RANK];
    {
        int64_t s = p->M * p->K;
        for (int d = ba - 1; d >= 0; --d) { a_own[d] = s; s *= a2[d]; }
        s = p->K * p->N;
        for (int d = bb - 1; d >= 0; --d) { b_own[d] = s; s *= b2[d]; }
    }
    p->batch_rank = r;
    p->batch = 1;
    for (int d = 0; d < r; ++d) {
        const int ia = d - (r - ba), ib = d - (r - bb);
        const int64_t da = ia >= 0 ? a2[ia] : 1;
        const int64_t db = ib >= 0 ? b2[ib] : 1;
        int64_t e;
        if (da == db) e = da;
        else if (da == 1) e = db;
        else if (db == 1) e = da;
        else { delete p; return OLC_ERR_BATCH_MISMATCH; }
        p->batch_shape[d] = e;
        // stride 0 wherever the operand's extent is 1 (broadcast or trivial)
        p->a_bstride[d] = (ia >= 0 && da != 1) ? a_own[ia] : 0;
        p->b_bstride[d] = (ib >= 0 && db != 1) ? b_own[ib] : 0;
        p->batch *= e;
    }

    // 3. output shape: batch + [M] (unless A was rank one) + [N] (unless B was)
    p->out_rank = 0;
    for (int d = 0; d < r; ++d) p->out_shape[p->out_rank++] = p->batch_shape[d];
    if (a_rank > 1) p->out_shape[p->out_rank++] = p->M;
    if (b_rank > 1) p->out_shape[p->out_rank++] = p->N;
    if (p->out_rank > OLC_MAX_RANK) { delete p; return OLC_ERR_RANK; }
    if (!tensor_fits(p->out_shape, p->out_rank, out_bytes(dtype))) { delete p; return OLC_ERR_INVALID; }

    // 4. collapse and fold the batch, then choose the algorithm
    collapse_and_fold(p);
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            sms > 0) {
            p->device = dev;
            p->sm_count = sms;
        }
    }
    cudaGetLastError();
    if (p->sm_count <= 0) p->sm_count = kDefaultSmCount;
    p->algo = choose_algorithm(p);
    p->forced = false;
    olc_status st = prepare_algorithm(p);
    if (st != OLC_OK) { delete p; return st; }
    *out = p;
    return OLC_OK;
}

olc_status olc_gemm_plan_create(const int64_t* a_shape, const int64_t* b_shape, int trans_a,
                                int trans_b, double alpha, double beta, const int64_t* c_shape,
                                int c_rank, olc_dtype dtype, olc_matmul_plan** out) {
    if (!out) return OLC_ERR_NULL;
    *out = nullptr;
    if (!a_shape || !b_shape || (c_rank > 0 && !c_shape)) return OLC_ERR_NULL;
    if (c_rank < -1 || c_rank > 2) return OLC_ERR_RANK;
    if (!valid_dtype(dtype) || is_fp8(dtype)) return OLC_ERR_DTYPE;   // Gemm: no 8-bit floats
    for (int i = 0; i < 2; ++i)
        if (a_shape[i] < 0 || b_shape[i] < 0) return OLC_ERR_NEGATIVE_DIM;
    for (int i = 0; i < c_rank; ++i)
        if (c_shape[i] < 0) return OLC_ERR_NEGATIVE_DIM;
    const int64_t M = trans_a ? a_shape[1] : a_shape[0];
    const int64_t K = trans_a ? a_shape[0] : a_shape[1];
    const int64_t Kb = trans_b ? b_shape[1] : b_shape[0];
    const int64_t N = trans_b ? b_shape[0] : b_shape[1];
    if (K != Kb) return OLC_ERR_K_MISMATCH;
    int64_t c2[2] = {1, 1};
    if (c_rank >= 1) c2[1] = c_shape[c_rank - 1];
    if (c_rank == 2) c2[0] = c_shape[0];
    if (c_rank >= 0 && (!(c2[0] == 1 || c2[0] == M) || !(c2[1] == 1 || c2[1] == N)))
        return OLC_ERR_BATCH_MISMATCH;   // C does not broadcast to [M, N]
    const int64_t y_shape[2] = {M, N};
    if (!tensor_fits(a_shape, 2, elem_bytes(dtype)) || !tensor_fits(b_shape, 2, elem_bytes(dtype)) ||
        !tensor_fits(y_shape, 2, elem_bytes(dtype)))
        return OLC_ERR_INVALID;

    olc_matmul_plan* p = new (std::nothrow) olc_matmul_plan;
    if (!p) return OLC_ERR_OOM;
    std::memset(p, 0, sizeof *p);
    p->dtype = dtype;
    p->a_rank = p->b_rank = 2;
    std::memcpy(p->a_shape, a_shape, sizeof(int64_t) * 2);
    std::memcpy(p->b_shape, b_shape, sizeof(int64_t) * 2);
    p->device = -1;
    p->M = M;
    p->N = N;
    p->K = K;
    p->batch = 1;
    p->batch_rank = 0;
    p->out_rank = 2;
    p->out_shape[0] = M;
    p->out_shape[1] = N;
    p->rows = M;
    p->items = 1;
    p->is_gemm = 1;
    p->trans_a = trans_a ? 1 : 0;
    p->trans_b = trans_b ? 1 : 0;
    p->alpha = alpha;
    p->beta = beta;
    p->c_rank = c_rank;
    p->c_shape[0] = c2[0];
    p->c_shape[1] = c2[1];
    p->c_rs = (c2[0] == 1) ? 0 : c2[1];
    p->c_cs = (c2[1] == 1) ? 0 : 1;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            sms > 0) {
            p->device = dev;
            p->sm_count = sms;
        }
    }
    cudaGetLastError();
    if (p->sm_count <= 0) p->sm_count = kDefaultSmCount;
    p->algo = choose_algorithm(p);
    olc_status st = prepare_algorithm(p);
    if (st != OLC_OK) { delete p; return st; }
    *out = p;
    return OLC_OK;
}

olc_status olc_gemm_execute(const olc_matmul_plan* plan, const void* A, const void* B,
                            const void* C, void* Y, void* stream) {
    if (!plan) return OLC_ERR_NULL;
    return run(plan, A, B, Y, static_cast<cudaStream_t>(stream), C);
}

void olc_matmul_plan_destroy(olc_matmul_plan* plan) {
    if (!plan) return;
    free_workspace(plan);
    free_stage(plan);
    if (plan->state_ev) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (plan->device >= 0 && cur != plan->device) cudaSetDevice(plan->device);
        cudaEventDestroy(plan->state_ev);
        if (plan->device >= 0 && cur >= 0 && cur != plan->device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    if (plan->pipe_ready) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (plan->device >= 0 && cur != plan->device) cudaSetDevice(plan->device);
        cudaStreamDestroy(plan->copy_in);
        cudaStreamDestroy(plan->copy_out);
        cudaEventDestroy(plan->ev_start);
        cudaEventDestroy(plan->ev_b);
        cudaEventDestroy(plan->ev_done);
        for (int i = 0; i < 8; ++i) {
            cudaEventDestroy(plan->ev_a[i]);
            cudaEventDestroy(plan->ev_y[i]);
        }
        if (plan->device >= 0 && cur >= 0 && cur != plan->device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    if (plan->const_b || plan->const_bt || plan->const_b_pad) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (plan->device >= 0 && cur != plan->device) cudaSetDevice(plan->device);
        if (plan->const_b) cudaFree(plan->const_b);
        if (plan->const_bt) cudaFree(plan->const_bt);
        if (plan->const_b_pad) cudaFree(plan->const_b_pad);
        if (plan->device >= 0 && cur >= 0 && cur != plan->device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    delete plan;
}

olc_status olc_matmul_plan_set_constant_b(olc_matmul_plan* plan, const void* B, int64_t b_numel,
                                          void* stream) {
    if (!plan) return OLC_ERR_NULL;
    const int64_t want = numel(plan->b_shape, plan->b_rank);
    if (b_numel != want) return OLC_ERR_BUFFER_TOO_SMALL;   // must be exactly the planned B
    if (want > 0 && !B) return OLC_ERR_NULL;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return from_cuda(cudaErrorNoDevice);
    if (plan->device >= 0 && cur != plan->device) return OLC_ERR_WRONG_DEVICE;
    if (plan->device < 0) {
        plan->device = cur;
        if ((plan->partial_bytes > 0 || plan->counter_count > 0) && !plan->workspace) {
            olc_status st = prepare_algorithm(plan);
            if (st != OLC_OK) return st;
        }
    }
    const size_t bytes = (size_t)(want * elem_bytes(plan->dtype));
    if (!plan->const_b || plan->const_b_bytes != bytes) {
        if (plan->const_b) cudaFree(plan->const_b);
        plan->const_b = nullptr;
        plan->const_b_bytes = 0;
        if (bytes > 0) {
            void* mem = nullptr;
            if (cudaMalloc(&mem, bytes) != cudaSuccess) {
                cudaGetLastError();
                return OLC_ERR_OOM;
            }
            plan->const_b = mem;
        }
        plan->const_b_bytes = bytes;
    }
    plan->const_b_set = 0;
    if (bytes > 0) {
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        // host or device source (unified addressing); the copy has completed
        // when this call returns, so the caller may free or reuse its buffer
        cudaError_t e = cudaMemcpyAsync(plan->const_b, B, bytes, cudaMemcpyDefault, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    // 8-bit float tensor-core plans: keep B transposed as well ([N, K], the
    // K-major operand the MMA reads), so executes with the constant B skip
    // the per-call transpose
    if (plan->const_bt) {
        cudaFree(plan->const_bt);
        plan->const_bt = nullptr;
        plan->const_bt_bytes = 0;
    }
    // 8-bit few-row plans (automatic kernel family): with a constant B the
    // tcgen05 kernel reads the transposed copy as loaded, streaming B at the
    // rate of the 16-bit swapped kernel, so the plan moves to it
    // (from 2 rows: one row streams faster on the SIMT kernel, 40.9 against
    // 42.5 us for [1, 8192] x [8192, 28672])
    plan->f8_const_tc = 0;
    if (bytes > 0 && is_fp8_tc_format(plan->dtype) && plan->algo == OLC_ALGO_SKINNY_M &&
        (plan->tc_variant == 3 || (plan->tc_variant == 0 && plan->rows >= 2))) {
        plan->f8_const_tc = 1;
        const Problem pr = make_problem(plan, nullptr, plan->const_b, nullptr);
        if (!f8_skinny_tc_ok(plan->dtype, pr)) plan->f8_const_tc = 0;
    }
    {
        const olc_status st = prepare_algorithm(plan);   // the kernel family sizes the workspace
        if (st != OLC_OK) return st;
    }
    if (bytes > 0 && is_fp8(plan->dtype) && (plan->algo == OLC_ALGO_GENERAL_TC || plan->f8_const_tc)) {
        Problem pr = make_problem(plan, nullptr, plan->const_b, nullptr);
        void* mem = nullptr;
        if (cudaMalloc(&mem, bytes) != cudaSuccess) {
            cudaGetLastError();
            return OLC_ERR_OOM;
        }
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        cudaError_t e = launch_fp8_transpose(pr, mem, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            cudaFree(mem);
            return from_cuda(e);
        }
        plan->const_bt = mem;
        plan->const_bt_bytes = bytes;
    }
    // 16-bit tensor-core plans whose B rows are not 16-byte multiples: keep
    // B with padded rows as well, the copy every execute would make
    if (plan->const_b_pad) {
        cudaFree(plan->const_b_pad);
        plan->const_b_pad = nullptr;
        plan->const_b_pad_bytes = 0;
    }
    const StoredRows rb = stored_b(plan);
    if (bytes > 0 && is_half(plan->dtype) && plan->algo == OLC_ALGO_GENERAL_TC && !plan->trans_b &&
        rb.cols % 8 != 0) {
        const size_t pbytes = (size_t)(rb.rows * pad8(rb.cols) * 2);
        void* mem = nullptr;
        if (cudaMalloc(&mem, pbytes) != cudaSuccess) {
            cudaGetLastError();
            return OLC_ERR_OOM;
        }
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        cudaError_t e = launch_pad_rows16(plan->const_b, mem, rb.rows, rb.cols, pad8(rb.cols), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            cudaFree(mem);
            return from_cuda(e);
        }
        plan->const_b_pad = mem;
        plan->const_b_pad_bytes = pbytes;
    }
    plan->const_b_set = 1;
    return OLC_OK;
}

int olc_matmul_plan_has_constant_b(const olc_matmul_plan* plan) {
    return plan && plan->const_b_set ? 1 : 0;
}

olc_status olc_matmul_execute_constant(const olc_matmul_plan* plan, const void* A, void* Y,
                                       void* stream) {
    if (!plan) return OLC_ERR_NULL;
    if (!plan->const_b_set) return OLC_ERR_NO_CONSTANT_B;
    return run(plan, A, plan->const_b, Y, static_cast<cudaStream_t>(stream));
}

olc_status olc_gemm_execute_constant(const olc_matmul_plan* plan, const void* A, const void* C,
                                     void* Y, void* stream) {
    if (!plan) return OLC_ERR_NULL;
    if (!plan->const_b_set) return OLC_ERR_NO_CONSTANT_B;
    return run(plan, A, plan->const_b, Y, static_cast<cudaStream_t>(stream), C);
}

olc_status olc_matmul_plan_set_epilogue(olc_matmul_plan* plan, int activation, int residual) {
    if (!plan) return OLC_ERR_NULL;
    if (activation < OLC_ACT_NONE || activation > OLC_ACT_GELU || residual < 0 || residual > 1)
        return OLC_ERR_INVALID;
    plan->act = activation;
    plan->residual = residual;
    return OLC_OK;
}

olc_status olc_matmul_execute_fused(const olc_matmul_plan* plan, const void* A, const void* B,
                                    const void* C, const void* R, void* Y, void* stream) {
    if (!plan) return OLC_ERR_NULL;
    if (!B && numel(plan->b_shape, plan->b_rank) > 0) {
        if (!plan->const_b_set) return OLC_ERR_NO_CONSTANT_B;
        B = plan->const_b;
    }
    if (plan->residual && !R && out_numel(plan) > 0) return OLC_ERR_NULL;
    return run(plan, A, B, Y, static_cast<cudaStream_t>(stream), C, R);
}

olc_status olc_matmul_execute(const olc_matmul_plan* plan, const void* A, const void* B, void* Y,
                              void* stream) {
    if (!plan) return OLC_ERR_NULL;
    return run(plan, A, B, Y, static_cast<cudaStream_t>(stream));
}

olc_status olc_matmul_execute_checked(const olc_matmul_plan* plan, const void* A, int64_t a_numel,
                                      const void* B, int64_t b_numel, void* Y, int64_t y_numel,
                                      void* stream) {
    if (!plan) return OLC_ERR_NULL;
    const int64_t n = out_numel(plan);
    if (n > 0) {
        if (y_numel < n) return OLC_ERR_BUFFER_TOO_SMALL;
        if (plan->K > 0) {
            if (a_numel < numel(plan->a_shape, plan->a_rank)) return OLC_ERR_BUFFER_TOO_SMALL;
            if (b_numel < numel(plan->b_shape, plan->b_rank)) return OLC_ERR_BUFFER_TOO_SMALL;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    olc_status st = run(plan, A, B, Y, s);
    if (st != OLC_OK || n == 0) return st;
    unsigned int flags = 0;
    cudaError_t e = read_and_clear_device_error(&flags, s);
    if (e != cudaSuccess) return from_cuda(e);
    return flags ? OLC_ERR_DEVICE_TIMEOUT : OLC_OK;
}

namespace {

// Row chunks of a host-buffer product that can be pipelined (copy in, compute
// and copy out of different chunks at once): one 2-D product (the batch, if
// any, folded into rows), a workspace-free algorithm, no residual, and enough
// rows for several tensor-core row tiles per chunk.  0 = not pipelined.
int host_chunks(const olc_matmul_plan* p) {
    if (p->items != 1 || p->K == 0 || p->residual || is_fp8(p->dtype)) return 0;
    // chunks read A and write Y in place: rows must be 16-byte multiples
    if (is_half(p->dtype) && (p->K % 8 != 0 || p->N % 8 != 0)) return 0;
    if (p->algo != OLC_ALGO_GENERAL_TC && p->algo != OLC_ALGO_GENERAL_SIMT) return 0;
    if (p->splits > 1) return 0;          // K-sliced plans use the workspace per launch
    if (p->is_gemm && (p->trans_a || (p->c_rank >= 0 && p->c_rs != 0))) return 0;
    const int64_t rows = p->rows;
    if (rows < 4 * 1024) return 0;
    return 4;
}

olc_status pipe_init(olc_matmul_plan* p) {
    if (p->pipe_ready) return OLC_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking);
    cudaEvent_t* evs[3] = {&p->ev_start, &p->ev_b, &p->ev_done};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&p->ev_a[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_y[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return from_cuda(e);
    p->pipe_ready = 1;
    return OLC_OK;
}

}  // namespace

olc_status olc_matmul_execute_host(const olc_matmul_plan* plan, const void* A_host,
                                   const void* B_host, void* Y_host, void* A_dev, void* B_dev,
                                   void* Y_dev, void* stream) {
    if (!plan) return OLC_ERR_NULL;
    const int64_t n = out_numel(plan);
    if (n == 0) return OLC_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t eb = elem_bytes(plan->dtype);
    if (!Y_host || !Y_dev) return OLC_ERR_NULL;
    const int chunks = aligned16(A_dev) && aligned16(B_dev) && aligned16(Y_dev) ? host_chunks(plan) : 0;
    if (chunks > 0) {
        if (!A_host || !B_host || !A_dev || !B_dev) return OLC_ERR_NULL;
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess) return from_cuda(cudaErrorNoDevice);
        if (plan->device >= 0 && cur != plan->device) return OLC_ERR_WRONG_DEVICE;
        olc_matmul_plan* mp = const_cast<olc_matmul_plan*>(plan);
        if (mp->device < 0) mp->device = cur;
        olc_status st = pipe_init(mp);
        if (st != OLC_OK) return st;
        // copy_in: B, then A in row chunks; the user stream computes chunk i
        // once its rows have arrived; copy_out returns chunk i's rows of Y
        // once they are computed; the user stream waits for the last copy.
        const int64_t rows = plan->rows, K = plan->K, N = plan->N;
        const int64_t step = (rows / chunks + 255) / 256 * 256;
        int whole_ways = 0;
        if (plan->algo == OLC_ALGO_GENERAL_TC && plan->tc_variant == 0) {
            const Problem whole = make_problem(plan, A_dev, B_dev, Y_dev);
            whole_ways = tc_general_csplit_ways(plan->dtype, whole, plan->sm_count);
        }
        const size_t b_bytes = (size_t)(numel(plan->b_shape, plan->b_rank) * eb);
        cudaError_t e = cudaEventRecord(mp->ev_start, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(mp->copy_in, mp->ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(mp->copy_out, mp->ev_start, 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(B_dev, B_host, b_bytes, cudaMemcpyHostToDevice, mp->copy_in);
        if (e == cudaSuccess) e = cudaEventRecord(mp->ev_b, mp->copy_in);
        int nc = 0;
        for (int64_t r0 = 0; r0 < rows && e == cudaSuccess; r0 += step, ++nc) {
            const int64_t rn = step < rows - r0 ? step : rows - r0;
            e = cudaMemcpyAsync(static_cast<unsigned char*>(A_dev) + r0 * K * eb,
                                static_cast<const unsigned char*>(A_host) + r0 * K * eb,
                                (size_t)(rn * K * eb), cudaMemcpyHostToDevice, mp->copy_in);
            if (e == cudaSuccess) e = cudaEventRecord(mp->ev_a[nc], mp->copy_in);
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, mp->ev_b, 0);
        nc = 0;
        for (int64_t r0 = 0; r0 < rows && e == cudaSuccess; r0 += step, ++nc) {
            const int64_t rn = step < rows - r0 ? step : rows - r0;
            e = cudaStreamWaitEvent(s, mp->ev_a[nc], 0);
            if (e != cudaSuccess) break;
            // chunk rows r0 .. r0 + rn of the same product (row-major A and Y)
            olc_matmul_plan sub = *plan;
            sub.rows = rn;
            sub.M = rn;
            // the chunks sum every element as the whole product would: the
            // same cluster split-K slices, or none
            sub.chunk_tc_ways = whole_ways >= 2 ? whole_ways : 1;
            const void* Ac = static_cast<const unsigned char*>(A_dev) + r0 * K * eb;
            void* Yc = static_cast<unsigned char*>(Y_dev) + r0 * N * eb;
            const void* Cc = nullptr;
            st = run(&sub, Ac, B_dev, Yc, s, Cc);
            if (st != OLC_OK) return st;
            e = cudaEventRecord(mp->ev_y[nc], s);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(mp->copy_out, mp->ev_y[nc], 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(static_cast<unsigned char*>(Y_host) + r0 * N * eb,
                                    static_cast<const unsigned char*>(Y_dev) + r0 * N * eb,
                                    (size_t)(rn * N * eb), cudaMemcpyDeviceToHost, mp->copy_out);
        }
        if (e == cudaSuccess) e = cudaEventRecord(mp->ev_done, mp->copy_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, mp->ev_done, 0);
        return from_cuda(e);
    }
    if (plan->K > 0) {
        if (!A_host || !B_host || !A_dev || !B_dev) return OLC_ERR_NULL;
        cudaError_t e = cudaMemcpyAsync(A_dev, A_host, numel(plan->a_shape, plan->a_rank) * eb,
                                        cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(B_dev, B_host, numel(plan->b_shape, plan->b_rank) * eb,
                                cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    olc_status st = run(plan, A_dev, B_dev, Y_dev, s);
    if (st != OLC_OK) return st;
    return from_cuda(cudaMemcpyAsync(Y_host, Y_dev, n * out_bytes(plan->dtype), cudaMemcpyDeviceToHost, s));
}

olc_status olc_matmul_plan_output_shape(const olc_matmul_plan* plan, int64_t* shape, int capacity,
                                        int* rank) {
    if (!plan || !rank || (!shape && plan->out_rank > 0)) return OLC_ERR_NULL;
    if (capacity < plan->out_rank) return OLC_ERR_INVALID;
    for (int i = 0; i < plan->out_rank; ++i) shape[i] = plan->out_shape[i];
    *rank = plan->out_rank;
    return OLC_OK;
}

olc_status olc_matmul_plan_dims(const olc_matmul_plan* plan, int64_t* M, int64_t* N, int64_t* K,
                                int64_t* batch) {
    if (!plan) return OLC_ERR_NULL;
    if (M) *M = plan->M;
    if (N) *N = plan->N;
    if (K) *K = plan->K;
    if (batch) *batch = plan->batch;
    return OLC_OK;
}

olc_status olc_matmul_plan_batch(const olc_matmul_plan* plan, int* batch_rank,
                                 int64_t* batch_shape, int64_t* a_strides, int64_t* b_strides) {
    if (!plan) return OLC_ERR_NULL;
    if (batch_rank) *batch_rank = plan->batch_rank;
    for (int d = 0; d < plan->batch_rank; ++d) {
        if (batch_shape) batch_shape[d] = plan->batch_shape[d];
        if (a_strides) a_strides[d] = plan->a_bstride[d];
        if (b_strides) b_strides[d] = plan->b_bstride[d];
    }
    return OLC_OK;
}

olc_status olc_matmul_plan_launch_shape(const olc_matmul_plan* plan, int64_t* rows,
                                        int64_t* items, int* collapsed_rank) {
    if (!plan) return OLC_ERR_NULL;
    if (rows) *rows = plan->rows;
    if (items) *items = plan->items;
    if (collapsed_rank) *collapsed_rank = plan->map.rank;
    return OLC_OK;
}

int olc_matmul_plan_algorithm(const olc_matmul_plan* plan) { return plan ? plan->algo : -1; }

olc_status olc_matmul_plan_force_algorithm(olc_matmul_plan* plan, int algo) {
    if (!plan) return OLC_ERR_NULL;
    if (algo == OLC_ALGO_AUTO) {
        plan->algo = choose_algorithm(plan);
        plan->forced = false;
        return prepare_algorithm(plan);
    }
    if (algo < OLC_ALGO_EMPTY || algo > OLC_ALGO_GENERAL_SIMT) return OLC_ERR_INVALID;
    const int n = (int)(out_numel(plan) > 0);
    if (!n || plan->K == 0) {
        if (algo != choose_algorithm(plan)) return OLC_ERR_ALIGNMENT;
    } else if (!feasible(plan, algo)) {
        return OLC_ERR_ALIGNMENT;
    }
    plan->algo = algo;
    plan->forced = true;
    return prepare_algorithm(plan);
}

int olc_matmul_plan_algorithm_for(const olc_matmul_plan* plan, const void* A, const void* B,
                                  const void* Y, const void* R) {
    if (!plan) return -1;
    return route_of(plan, A, B, Y, R).algo;
}

int olc_matmul_plan_staging_copies(const olc_matmul_plan* plan, const void* A, const void* B,
                                   const void* Y, const void* R) {
    if (!plan) return -1;
    const Route r = route_of(plan, A, B, Y, R);
    return (r.need.a ? 1 : 0) + (r.need.b ? 1 : 0);
}

olc_status olc_matmul_plan_set_splits(olc_matmul_plan* plan, int splits) {
    if (!plan) return OLC_ERR_NULL;
    if (splits < 0 || splits > 4096) return OLC_ERR_INVALID;
    plan->split_hint = splits;
    return prepare_algorithm(plan);
}

int olc_matmul_plan_splits(const olc_matmul_plan* plan) { return plan ? plan->splits : -1; }

olc_status olc_matmul_plan_set_tc_variant(olc_matmul_plan* plan, int variant) {
    if (!plan) return OLC_ERR_NULL;
    if (variant < 0 || variant > 3) return OLC_ERR_INVALID;
    plan->tc_variant = variant;
    return prepare_algorithm(plan);   // the workspace depends on the kernel family
}

int olc_matmul_plan_launches(const olc_matmul_plan* plan) {
    if (!plan) return -1;
    if (plan->algo == OLC_ALGO_EMPTY) return 0;
    int n = 1;
    if (plan->algo == OLC_ALGO_GENERAL_TC && is_half(plan->dtype)) {
        // staging copies of rows that are not 16-byte multiples
        const StageNeed need = stage_need(plan, nullptr, nullptr, true, plan->const_b_pad != nullptr);
        n += (need.a ? 1 : 0) + (need.b ? 1 : 0);
    }
    if (plan->algo == OLC_ALGO_GENERAL_TC && is_fp8(plan->dtype) && !plan->const_bt) ++n;   // B transpose
    return n;
}

size_t olc_matmul_plan_workspace_bytes(const olc_matmul_plan* plan) {
    return plan ? plan->ws_bytes : 0;
}

int olc_matmul_plan_describe(const olc_matmul_plan* plan, char* buf, size_t cap) {
    if (!plan) return -1;
    char tmp[512];
    char slices[48] = "";
    if (plan->cluster_slices > 1)
        std::snprintf(slices, sizeof slices, " cluster_slices=%d", plan->cluster_slices);
    int n = std::snprintf(tmp, sizeof tmp,
                          "algo=%s dtype=%d M=%lld N=%lld K=%lld batch=%lld rows=%lld items=%lld "
                          "collapsed_rank=%d splits=%d%s ws=%zu sms=%d%s",
                          olc_algorithm_name(plan->algo), (int)plan->dtype, (long long)plan->M,
                          (long long)plan->N, (long long)plan->K, (long long)plan->batch,
                          (long long)plan->rows, (long long)plan->items, plan->map.rank,
                          plan->splits, slices, plan->ws_bytes, plan->sm_count,
                          plan->forced ? " forced" : "");
    if (buf && cap > 0) {
        std::strncpy(buf, tmp, cap - 1);
        buf[cap - 1] = '\0';
    }
    return n;
}

const char* olc_status_string(int status) {
    switch (status) {
        case OLC_OK: return "ok";
        case OLC_ERR_NULL: return "null pointer argument";
        case OLC_ERR_RANK: return "rank out of range (1..8)";
        case OLC_ERR_NEGATIVE_DIM: return "negative dimension";
        case OLC_ERR_K_MISMATCH: return "inner dimensions differ";
        case OLC_ERR_BATCH_MISMATCH: return "batch dimensions do not broadcast";
        case OLC_ERR_DTYPE: return "unsupported element type";
        case OLC_ERR_ALIGNMENT: return "algorithm cannot take this shape or type";
        case OLC_ERR_BUFFER_TOO_SMALL: return "buffer smaller than the planned tensor";
        case OLC_ERR_NO_CONSTANT_B: return "plan owns no constant B";
        case OLC_ERR_CUDA: return "CUDA runtime error";
        case OLC_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case OLC_ERR_OOM: return "out of memory";
        case OLC_ERR_INVALID: return "invalid argument";
        case OLC_ERR_WRONG_DEVICE: return "current device is not the plan's device";
        case OLC_ERR_SCRATCH_LIMIT: return "problem needs more than the static scratch array";
        case OLC_ERR_NEEDS_RESIDUAL: return "plan fuses a residual: execute with olc_matmul_execute_fused";
    }
    return "unknown status";
}

const char* olc_algorithm_name(int algo) {
    switch (algo) {
        case OLC_ALGO_AUTO: return "auto";
        case OLC_ALGO_EMPTY: return "empty";
        case OLC_ALGO_ZERO_FILL: return "zero_fill";
        case OLC_ALGO_DIRECT: return "direct";
        case OLC_ALGO_SKINNY_M: return "skinny_m";
        case OLC_ALGO_SKINNY_N: return "skinny_n";
        case OLC_ALGO_SPLIT_K: return "split_k";
        case OLC_ALGO_GENERAL_TC: return "general_tc";
        case OLC_ALGO_GENERAL_SIMT: return "general_simt";
    }
    return "unknown";
}

int olc_version(void) { return 100; }

}  // extern "C"
