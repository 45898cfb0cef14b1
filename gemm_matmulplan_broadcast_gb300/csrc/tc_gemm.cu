// GENERAL_TC: tcgen05 tensor-core GEMM for FLOAT16 / BFLOAT16 on sm_103a.
//
// "MatMul Kernel Design", section "Types and algorithm selection": FLOAT16
// and BFLOAT16 accumulate in float32 and narrow once at the end; "Gemm and
// MatMul Performance Roadmap", section "Phase 3: native low-precision
// kernels": no full-tensor widening on any path -- here A and B stay 16-bit
// from HBM to the tensor core, the float32 accumulator lives in tensor memory
// (TMEM), and only the epilogue narrows.  The pages' five-loop CPU blocking
// (section "Target computation algorithm": packed B panel reused by every row
// block, packed A panel reused by every column micro-panel, the C tile kept in
// registers for the whole reduction) maps onto:
//
//   output tile 128 x 256 per CTA   <- TMA 2-D tiles of A (128 x 64) and B
//   (64 x 256) staged through a 4-deep shared-memory ring, consumed by
//   tcgen05.mma (M=128, N=256, K=16) into a 128 x 256 float32 accumulator in
//   TMEM, which stays there for the whole K loop.
//
// Warp roles (6 warps, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one lane): waits for a free stage, arms its
//               mbarrier with the byte count, issues the A and B tile loads;
//   warp 1      MMA issuer (one lane) and TMEM owner: waits for a full stage,
//               issues 4 MMAs, commits the stage back to the producer; after
//               a tile's last K block commits the accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes (= 32 output
//               rows), round-to-nearest-even narrowing, 16-byte stores.
// The two TMEM accumulators (2 x 256 columns = all 512) let the epilogue of
// tile i overlap the MMAs of tile i+1.
//
// Operand layouts in shared memory (both 128-byte swizzled, as TMA writes
// them): A is K-major (rows of 64 K-elements = 128 bytes, 8-row groups 1024
// bytes apart); B stays MN-major as it is in HBM (row-major [K, N]): each
// stage holds four 64-column blocks of 64 K-rows, 8192 bytes apart, each
// K-row 128 bytes.  The MMA reads B through the "transpose B" bit of the
// instruction descriptor, so no transposed copy of B is ever made.
//
// Every mbarrier wait is bounded (about 4 s of %globaltimer).  A wait that
// runs out sets the library's device error word and an abort flag that every
// role polls; the CTA then waits (bounded) for its own TMA loads and MMAs in
// flight, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace olc {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;               // one 128-byte swizzle span of 16-bit A elements
constexpr int UMMA_K = 16;
constexpr int A_STAGE_BYTES = BM * BK * 2;       // 16 KiB
constexpr int STAGE_BUDGET = 192 * 1024;         // shared memory for the stage ring
constexpr int MAX_STAGES = 12;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;                 // warps 2..5
constexpr int GROUP_M = 16;                      // tile raster: 16 M-blocks per group
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // default bound of every wait
constexpr int SUM_BATCH = 12;                    // partials loaded per reduction round trip

// Per tile width BN: how B (MN-major, N contiguous) is staged.  A 64-deep
// stage of B is cut into boxes BLK_COLS columns wide whose rows are one
// swizzle span: 128-byte swizzle with 64-column boxes for BN >= 64, 64-byte
// swizzle for BN = 32, 32-byte swizzle for BN = 16.
template <int BN>
struct Cfg {
    static constexpr int SW = BN >= 64 ? 128 : BN * 2;        // swizzle span in bytes
    static constexpr int BLK_COLS = SW / 2;
    static constexpr int NBLK = BN / BLK_COLS;
    static constexpr int B_BLK_BYTES = BK * SW;               // one box: BK rows of SW bytes
    static constexpr int B_STAGE_BYTES = NBLK * B_BLK_BYTES;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGES =
        STAGE_BUDGET / STAGE_BYTES > MAX_STAGES ? MAX_STAGES : STAGE_BUDGET / STAGE_BYTES;
    static constexpr uint32_t LAYOUT = SW == 128 ? 2u : (SW == 64 ? 4u : 6u);   // descriptor code
    static constexpr int ACC_COLS = BN;
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* alignment slack */ + 512;
    static_assert(STAGE_BYTES % 1024 == 0, "stage buffers must keep 1024-byte alignment");
    static_assert(BN % BLK_COLS == 0, "tile width must be whole boxes");
};

struct Smem {
    // stage buffers come first (1024-byte aligned), barriers after
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int last_flag;
};

struct Params {
    int64_t M, N, K;          // per batch item
    int64_t items;
    int64_t tiles_m, tiles_n, tiles_per_item, total_tiles;
    int64_t k_blocks;         // BK-deep blocks of the whole K
    int64_t a_item_elems;     // M * K: A matrix size (for the TMA batch coordinate)
    int64_t b_item_elems;     // K * N
    BatchMap map;
    void* Y;
    unsigned int* err;
    int is_bf16;
    // split-K (splits == 1 and null pointers otherwise)
    int splits;               // K slices per tile
    int group;                // slices per first-level reduction group
    int groups;               // ceil(splits / group)
    int64_t kb_per_split;     // k-blocks per slice
    uint32_t stage_tx_bytes;  // bytes the TMA loads of one stage deliver
    int stream;               // 1: stream-K shares (split instantiation only)
    int a_mn;                 // A stored [K, M] (Gemm transA): MN-major A operand
    int b_k;                  // B stored [N, K] (Gemm transB): K-major B operand
    int y_unaligned;          // Y rows not 16-byte aligned: stores by alignment (general kernels)
    int b_blocks;             // CTA pairs, MN-major B with N a multiple of 64: tmap_b is the 4-D
                              // view [items][N/64][K][64] and one load brings both 64-column blocks
    int64_t pair_half_tiles;  // CTA pairs: the last tiles, run as two 256 x 128 halves each (a
                              // last partial wave of at most half the clusters); 0: none
    int f8_fmt;               // 8-bit float operands (pair kernel): 0 = E4M3, 1 = E5M2
    Epilogue epi;
    int64_t iterations;       // stream-K: total (tile, K block) iterations
    float* part1;             // [tiles][splits][BM][BN] float32 partial tiles
    float* part2;             // [tiles][groups][BM][BN] group sums
    unsigned int* cnt1;       // [tiles][groups] arrivals per group
    unsigned int* cnt2;       // [tiles] arrivals of group sums
};

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false when the wait ran out (after `limit_ns` of
// %globaltimer; the error word gets kErrWaitTimeout) or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            raise_device_error(err, kErrWaitTimeout);
            return false;
        }
    }
}

// Bounded wait used while draining after an abort (no abort check).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) return;
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (base lane + t), columns c .. c+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// the four epilogue warps only (named barrier 1)
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory");
}

// ---------------------------------------------------------------------------
// descriptors (host and device agree on these encodings; the host unit test
// checks them bit by bit)

// Shared-memory matrix descriptor for tcgen05: start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// the fixed value 1 in bits 46-47, base offset 0 in 49-51, relative LBO mode
// (bit 52 = 0), swizzle mode in 61-63 (2 = 128-byte, 4 = 64-byte, 6 = 32-byte).
__host__ __device__ constexpr uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                                 uint32_t layout) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
           ((uint64_t)(layout & 7u) << 61);
}

// Instruction descriptor for kind::f16: float32 accumulator (bits 4-5 = 1),
// A and B type in bits 7-9 / 10-12 (0 = F16, 1 = BF16), A major-ness in bit 15
// and B major-ness in bit 16 (0 = K-major, 1 = MN-major), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(int is_bf16, int m, int n, int a_mn_major,
                                                  int b_mn_major) {
    return (1u << 4) | ((uint32_t)is_bf16 << 7) | ((uint32_t)is_bf16 << 10) |
           ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// tile raster: groups of GROUP_M M-blocks, M fastest inside a group, so the
// tiles running at the same time share A row blocks and B column blocks in L2

__device__ __forceinline__ void tile_coords(const Params& p, int64_t t, int64_t& item,
                                            int64_t& mb, int64_t& nb) {
    item = t / p.tiles_per_item;
    const int64_t r = t % p.tiles_per_item;
    const int64_t group_span = (int64_t)GROUP_M * p.tiles_n;
    const int64_t g = r / group_span;
    const int64_t first_m = g * GROUP_M;
    const int64_t gm = min64(p.tiles_m - first_m, GROUP_M);
    const int64_t in = r % group_span;
    mb = first_m + in % gm;
    nb = in / gm;
}

// The work of one CTA as a sequence of pieces (tile, K blocks kb0..kb1-1).
// Unit mode: unit u = tile u / splits, slice u % splits, units dealt round
// robin over the CTAs.  Stream-K mode: the tiles' K blocks laid end to end
// form `iterations` steps; CTA c takes steps [c*I/G, (c+1)*I/G) and cuts them
// at tile boundaries.  A tile cut between CTAs has `parts` contributors;
// `slice` is this CTA's position among them (in K order).
struct Cursor {
    int64_t u;
    int64_t it, it_end;
};

__device__ __forceinline__ int64_t share_begin(const Params& p, int64_t c) {
    return c * p.iterations / (int64_t)gridDim.x;
}

// the CTA whose share holds step i
__device__ __forceinline__ int64_t owner_of(const Params& p, int64_t i) {
    int64_t c = i * (int64_t)gridDim.x / p.iterations;
    while (c + 1 < (int64_t)gridDim.x && share_begin(p, c + 1) <= i) ++c;
    while (c > 0 && share_begin(p, c) > i) --c;
    return c;
}

__device__ __forceinline__ Cursor cursor_begin(const Params& p) {
    Cursor c;
    c.u = blockIdx.x;
    c.it = p.stream ? share_begin(p, blockIdx.x) : 0;
    c.it_end = p.stream ? share_begin(p, blockIdx.x + 1) : 0;
    return c;
}

__device__ __forceinline__ bool cursor_next(const Params& p, Cursor& c, int64_t& tile, int& slice,
                                            int64_t& kb0, int64_t& kb1, int& parts) {
    if (!p.stream) {
        if (c.u >= p.total_tiles * p.splits) return false;
        tile = c.u / p.splits;
        slice = (int)(c.u % p.splits);
        kb0 = (int64_t)slice * p.kb_per_split;
        kb1 = min64(p.k_blocks, kb0 + p.kb_per_split);
        parts = p.splits;
        c.u += gridDim.x;
        return true;
    }
    if (c.it >= c.it_end) return false;
    tile = c.it / p.k_blocks;
    kb0 = c.it % p.k_blocks;
    kb1 = min64(p.k_blocks, kb0 + (c.it_end - c.it));
    c.it += kb1 - kb0;
    const int64_t first = owner_of(p, tile * p.k_blocks);
    const int64_t last = owner_of(p, (tile + 1) * p.k_blocks - 1);
    slice = (int)(blockIdx.x - first);
    parts = (int)(last - first + 1);
    return true;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int is_bf16) {
    if (is_bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float widen16(unsigned bits, bool is_bf16) {
    bits &= 0xFFFFu;
    return is_bf16 ? __uint_as_float(bits << 16) : __half2float(__ushort_as_half((unsigned short)bits));
}

// The epilogue on one float32 accumulator of output (i, j) within its item:
// alpha * acc + beta * C (C of the 16-bit output type), plus the residual
// whose 16-bit pattern is `rbits` (used when epi.R is set), then the
// activation; the plain product when epi.mode == 0.
__device__ __forceinline__ float tc_epi(const Params& p, float acc, int64_t i, int64_t j,
                                        unsigned rbits = 0) {
    if (p.epi.mode == 0) return acc;
    float y = __fmul_rn(p.epi.alpha_f, acc);
    if (p.epi.C) {
        const unsigned short bits =
            __ldg(static_cast<const unsigned short*>(p.epi.C) + i * p.epi.c_rs + j * p.epi.c_cs);
        y = __fadd_rn(y, __fmul_rn(p.epi.beta_f, widen16(bits, p.is_bf16)));
    }
    if (p.epi.R) y = __fadd_rn(y, widen16(rbits, p.is_bf16));
    return activate(p.epi.act, y);
}

// Residual pattern of the 16-bit output element at y (0 without a residual).
__device__ __forceinline__ unsigned resid16(const Params& p, const unsigned short* y) {
    return p.epi.R ? (unsigned)__ldg(residual_at(p.epi, y)) : 0u;
}

// The epilogue over one run of 2*NP accumulators (raw float32 bits in r) of
// output row `row`, columns col.., narrowed into NP packed pairs.  `dst` is
// the run's address in Y; the residual is read from the same offset in R,
// in the `groups` 16-byte groups the store will write.  Each step is one
// loop over the run behind a uniform test, so only the steps a plan uses
// are executed and the unrolled code stays small.
template <int NP>
__device__ __forceinline__ void epi_run(const Params& p, const uint32_t* r, int64_t row,
                                        int64_t col, const unsigned char* dst, int groups,
                                        uint32_t* packed) {
    float v[2 * NP];
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) v[i] = __uint_as_float(r[i]);
    if (p.epi.mode != 0) {
        const float alpha = p.epi.alpha_f;
        if (alpha != 1.0f) {
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i) v[i] = __fmul_rn(alpha, v[i]);
        }
        if (p.epi.C) {
            const unsigned short* c = static_cast<const unsigned short*>(p.epi.C) + row * p.epi.c_rs;
            const float beta = p.epi.beta_f;
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i)
                v[i] = __fadd_rn(v[i], __fmul_rn(beta, widen16(__ldg(c + (col + i) * p.epi.c_cs), p.is_bf16)));
        }
        if (p.epi.R && !p.y_unaligned) {
            const uint4* src = reinterpret_cast<const uint4*>(dst + p.epi.r_delta);
            uint32_t rr[NP];
#pragma unroll
            for (int q = 0; q < NP / 4; ++q) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (q < groups) w = __ldg(src + q);
                rr[4 * q] = w.x; rr[4 * q + 1] = w.y; rr[4 * q + 2] = w.z; rr[4 * q + 3] = w.w;
            }
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i)
                v[i] = __fadd_rn(v[i], widen16(rr[i >> 1] >> (16 * (i & 1)), p.is_bf16));
        } else if (p.epi.R) {
            // unaligned rows: the residual element by element (`groups` is
            // then the number of valid columns of the run)
            const unsigned short* src = reinterpret_cast<const unsigned short*>(dst + p.epi.r_delta);
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i)
                if (i < groups) v[i] = __fadd_rn(v[i], widen16(__ldg(src + i), p.is_bf16));
        }
        if (p.epi.act == OLC_ACT_RELU) {
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i) v[i] = v[i] < 0.f ? 0.f : v[i];
        } else if (p.epi.act == OLC_ACT_GELU) {
#pragma unroll
            for (int i = 0; i < 2 * NP; ++i) v[i] = gelu_f32(v[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) packed[i] = pack2(v[2 * i], v[2 * i + 1], p.is_bf16);
}

// Ask L2 for the residual of one output row run (cols columns from (row,
// col0) of item `item`), so the epilogue's residual loads hit L2.  The run
// starts on a 16-byte boundary and is a whole number of 16-byte groups
// (N is a multiple of 8 on the tensor-core path).
__device__ __forceinline__ void prefetch_residual(const Params& p, int64_t item, int64_t row,
                                                  int64_t col0, int64_t cols) {
    if (!p.epi.R || cols <= 0 || p.y_unaligned) return;
    const unsigned char* src = static_cast<const unsigned char*>(p.epi.R) +
                               ((item * p.M + row) * p.N + col0) * 2;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)(cols * 2))
                 : "memory");
}

// Sum `count` float32 partial tiles (`stride` floats apart) in order 0, 1,
// ... for the float4s at indices e0 and e1 (e1 < 0: only e0).  All loads of
// a batch of up to SUM_BATCH partials are issued before any is added, so a
// group costs one round trip to L2 instead of one per partial.
__device__ __noinline__ void ordered_sum4x2(const float* base, int64_t stride, int count,
                                            int64_t e0, int64_t e1, float4& r0, float4& r1) {
    const int64_t e1c = e1 >= 0 ? e1 : e0;   // branch-free loads; r1 unused when e1 < 0
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 a1 = a0;
    for (int s0 = 0; s0 < count; s0 += SUM_BATCH) {
        const int n = count - s0 < SUM_BATCH ? count - s0 : SUM_BATCH;
        float4 v0[SUM_BATCH], v1[SUM_BATCH];
#pragma unroll
        for (int j = 0; j < SUM_BATCH; ++j) {
            const int jj = j < n ? j : 0;
            const float4* src = reinterpret_cast<const float4*>(base + (int64_t)(s0 + jj) * stride);
            v0[j] = __ldcg(src + e0);
            v1[j] = __ldcg(src + e1c);
        }
#pragma unroll
        for (int j = 0; j < SUM_BATCH; ++j) {
            if (j < n) {
                a0.x += v0[j].x; a0.y += v0[j].y; a0.z += v0[j].z; a0.w += v0[j].w;
                a1.x += v1[j].x; a1.y += v1[j].y; a1.z += v1[j].z; a1.w += v1[j].w;
            }
        }
    }
    r0 = a0;
    r1 = a1;
}

// ---------------------------------------------------------------------------
// Stores of one 32-column run of 16-bit outputs (element i of the run in half
// i & 1 of packed[i >> 1]) to a row of Y that need not be 16-byte aligned:
// the general kernels with an odd N, or a Y pointer off a 16-byte boundary.
// A full run takes H single elements up to the next 16-byte boundary (pairs
// as 32-bit stores where the address allows), 16-byte stores of the shifted
// elements, then the rest; H is the run's start in elements modulo 8, so each
// of the 8 cases is unrolled with static register indices.

__device__ __forceinline__ uint32_t run_pair(const uint32_t (&pk)[16], int e) {
    // elements e and e + 1 packed (e static after unrolling)
    return (e & 1) ? __funnelshift_r(pk[e >> 1], pk[(e >> 1) + 1], 16) : pk[e >> 1];
}
__device__ __forceinline__ unsigned short run_elem(const uint32_t (&pk)[16], int e) {
    return (unsigned short)(pk[e >> 1] >> (16 * (e & 1)));
}

template <int H>
__device__ __forceinline__ void store_run_shifted(unsigned short* dst, const uint32_t (&pk)[16]) {
    constexpr int G = (32 - H) / 8;              // whole 16-byte groups after the head
    // head: elements 0..H-1 (dst + H is 16-byte aligned)
    if constexpr (H & 1) {
        dst[0] = run_elem(pk, 0);
#pragma unroll
        for (int e = 1; e < H; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = run_pair(pk, e);
    } else {
#pragma unroll
        for (int e = 0; e < H; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = run_pair(pk, e);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int e = H + 8 * g;
        *reinterpret_cast<uint4*>(dst + e) =
            make_uint4(run_pair(pk, e), run_pair(pk, e + 2), run_pair(pk, e + 4), run_pair(pk, e + 6));
    }
    // tail: elements H + 8 G .. 31, starting on a 16-byte boundary
#pragma unroll
    for (int e = H + 8 * G; e + 1 < 32; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = run_pair(pk, e);
    if constexpr (((32 - H - 8 * G) & 1) != 0) dst[31] = run_elem(pk, 31);
}

// `valid` (1..32) elements of the run to dst (2-byte aligned).
__device__ __forceinline__ void store_run_unaligned(unsigned char* dst_bytes, const uint32_t (&pk)[16],
                                                    int valid) {
    unsigned short* dst = reinterpret_cast<unsigned short*>(dst_bytes);
    if (valid < 32) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            if (e < valid) dst[e] = run_elem(pk, e);
        return;
    }
    const int h = (int)((8 - ((reinterpret_cast<uintptr_t>(dst) >> 1) & 7)) & 7);
    switch (h) {
        case 0: store_run_shifted<0>(dst, pk); break;
        case 1: store_run_shifted<1>(dst, pk); break;
        case 2: store_run_shifted<2>(dst, pk); break;
        case 3: store_run_shifted<3>(dst, pk); break;
        case 4: store_run_shifted<4>(dst, pk); break;
        case 5: store_run_shifted<5>(dst, pk); break;
        case 6: store_run_shifted<6>(dst, pk); break;
        default: store_run_shifted<7>(dst, pk); break;
    }
}

// Narrow four float32 sums and store them at output row r, column col of
// the tile (col < N checked by the caller).
__device__ __forceinline__ void store4(const Params& p, int64_t item, int64_t row, int64_t col,
                                       float4 v) {
    unsigned short* y = static_cast<unsigned short*>(p.Y) + (item * p.M + row) * p.N + col;
    uint2 rr = make_uint2(0u, 0u);
    if (p.epi.R) rr = __ldg(reinterpret_cast<const uint2*>(residual_at(p.epi, y)));
    v.x = tc_epi(p, v.x, row, col, rr.x);
    v.y = tc_epi(p, v.y, row, col + 1, rr.x >> 16);
    v.z = tc_epi(p, v.z, row, col + 2, rr.y);
    v.w = tc_epi(p, v.w, row, col + 3, rr.y >> 16);
    *reinterpret_cast<uint2*>(y) = make_uint2(pack2(v.x, v.y, p.is_bf16), pack2(v.z, v.w, p.is_bf16));
}

// Swapped operands: the tile holds Y^T (TMEM lane = output column n, TMEM
// column = output row m); store four consecutive rows m0..m0+3 of column n.
__device__ __forceinline__ void store4_t(const Params& p, int64_t item, int64_t n, int64_t m0,
                                         float4 v) {
    const float f[4] = {v.x, v.y, v.z, v.w};
    unsigned short* y = static_cast<unsigned short*>(p.Y);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (m0 + i < p.M) {
            unsigned short* yp = y + (item * p.M + m0 + i) * p.N + n;
            const uint32_t h = pack2(tc_epi(p, f[i], m0 + i, n, resid16(p, yp)), 0.f, p.is_bf16);
            *yp = (unsigned short)(h & 0xFFFFu);
        }
    }
}

template <int BN, bool SPLIT, bool SWAP>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_b, const Params p) {
    using C = Cfg<BN>;
    constexpr int STAGES = C::STAGES;
    constexpr int CH = BN < 32 ? BN : 32;             // accumulator columns per tcgen05.ld
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned stage buffers (every swizzle pattern repeats within
    // 1024 bytes and the descriptors assume an aligned base)
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem* s = reinterpret_cast<Smem*>(base + STAGES * C::STAGE_BYTES);
    volatile int* abort_flag = &s->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s->acc_full[i], 1);
            mbar_init(&s->acc_empty[i], 4);   // one arrival per epilogue warp
        }
        mbar_init(&s->drain, 1);
        s->abort_flag = 0;
        s->last_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // barriers visible to every warp; the producer starts loading right away
    // while warp 1 allocates TMEM and hands the address to the epilogue warps
    // through named barrier 2 (warps 1..5)
    __syncthreads();
    grid_dependency_wait();
    grid_launch_dependents();
    uint32_t tmem_base = 0;
    if (warp == 1) tmem_alloc(&s->tmem_base, C::TMEM_COLS);
    if (warp >= 1) {
        tc_fence_before();
        asm volatile("bar.sync 2, %0;" ::"n"(THREADS - 32) : "memory");
        tc_fence_after();
        tmem_base = s->tmem_base;
    }

    // one reduced float4 of a tile (entries e4*4 .. e4*4+3 of the BM x BN
    // partial layout) to Y
    auto store_sum = [&](int64_t item, int64_t mb, int64_t nb, int64_t e4, float4 v) {
        const int64_t r = (e4 * 4) / BN, cc = (e4 * 4) % BN;
        if constexpr (SWAP) {
            store4_t(p, item, mb * BM + r, cc, v);
        } else {
            if (nb * BN + cc < p.N) store4(p, item, mb * BM + r, nb * BN + cc, v);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            // running shared addresses and register bitmasks keep the issue
            // loop short (see the pair kernel's producer)
            const uint32_t stage0 = smem_u32(base);
            const uint32_t full0 = smem_u32(&s->full[0]);
            uint32_t stage = 0, phase = 0, armed_bits = 0, parity_bits = 0;
            bool ok = true;
            Cursor cur = cursor_begin(p);
            int64_t tile, kb0, kb1;
            int slice, parts;
            while (ok && cursor_next(p, cur, tile, slice, kb0, kb1, parts)) {
                int64_t item, mb, nb;
                tile_coords(p, tile, item, mb, nb);
                int64_t a_off, b_off;
                batch_offsets(p.map, item, a_off, b_off);
                const int a_item = (int)(a_off / p.a_item_elems);
                const int b_item = (int)(b_off / p.b_item_elems);
                const int m0 = (int)(mb * BM), n0 = (int)(nb * BN);
                int k0 = (int)(kb0 * BK);
                for (int64_t kb = kb0; kb < kb1; ++kb, k0 += BK) {
                    if (!mbar_wait(&s->empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    const uint32_t sa = stage0 + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    const uint32_t fb = full0 + stage * (uint32_t)sizeof(uint64_t);
                    mbar_arrive_expect_tx(&s->full[stage], p.stage_tx_bytes);
                    armed_bits |= 1u << stage;
                    parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    if constexpr (!SWAP) {
                        if (!p.a_mn) {
                            tma_load_3d(sa, &tmap_a, fb, k0, m0, a_item);
                        } else {
                            // A stored [K, M]: two MN-major 64-row boxes
                            tma_load_3d(sa, &tmap_a, fb, m0, k0, a_item);
                            tma_load_3d(sa + 64 * BK * 2, &tmap_a, fb, m0 + 64, k0, a_item);
                        }
                        if (!p.b_k) {
#pragma unroll
                            for (int j = 0; j < C::NBLK; ++j)
                                tma_load_3d(sb + j * C::B_BLK_BYTES, &tmap_b, fb, n0 + C::BLK_COLS * j, k0,
                                            b_item);
                        } else {
                            // B stored [N, K]: one K-major box of BN rows
                            tma_load_3d(sb, &tmap_b, fb, k0, n0, b_item);
                        }
                    } else {
                        // MMA operand A = 128 columns of the problem's B (two
                        // 64-column MN-major boxes); operand B = the problem's
                        // A rows (K-major, rows past M read as zeros)
                        tma_load_3d(sa, &tmap_a, fb, m0, k0, b_item);
                        tma_load_3d(sa + 64 * BK * 2, &tmap_a, fb, m0 + 64, k0, b_item);
                        tma_load_3d(sb, &tmap_b, fb, k0, 0, a_item);
                        (void)n0;
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (*abort_flag) {
                // let this CTA's own loads land before the CTA goes away
                for (int i = 0; i < STAGES; ++i)
                    if ((armed_bits >> i) & 1u) mbar_wait_drain(&s->full[i], (parity_bits >> i) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = SWAP ? instr_desc(p.is_bf16, BM, BN, 1, 0)
                                        : instr_desc(p.is_bf16, BM, BN, p.a_mn, p.b_k ? 0 : 1);
            // descriptors of stage 0, advanced by adds to the start-address
            // field (see the pair kernel's MMA issuer).
            // Not swapped: A K-major (128-byte swizzle, 16 elements = 32
            // bytes per step) or MN-major (16 K-rows of 128 bytes per step,
            // the two 64-row boxes 8192 bytes apart); B MN-major (16 K-rows
            // of SW bytes per step, boxes of BLK_COLS columns B_BLK_BYTES
            // apart, 8-row groups 8 * SW apart) or K-major (transB: rows of
            // 64 K-elements).  Swapped: A = the problem's B, MN-major; B =
            // the problem's A rows, K-major.
            const uint32_t stage0 = smem_u32(base);
            uint64_t a_desc0, b_desc0, a_step, b_step;
            if constexpr (!SWAP) {
                a_desc0 = p.a_mn ? smem_desc(stage0, 64 * BK * 2, 1024, 2u) : smem_desc(stage0, 16, 1024, 2u);
                a_step = p.a_mn ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
                b_desc0 = p.b_k ? smem_desc(stage0 + A_STAGE_BYTES, 16, 1024, 2u)
                                : smem_desc(stage0 + A_STAGE_BYTES, C::B_BLK_BYTES, 8 * C::SW, C::LAYOUT);
                b_step = p.b_k ? (UMMA_K * 2) >> 4 : (UMMA_K * C::SW) >> 4;
            } else {
                a_desc0 = smem_desc(stage0, 64 * BK * 2, 1024, 2u);
                a_step = (UMMA_K * 128) >> 4;
                b_desc0 = smem_desc(stage0 + A_STAGE_BYTES, 16, 1024, 2u);
                b_step = (UMMA_K * 2) >> 4;
            }
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            Cursor cur = cursor_begin(p);
            int64_t tile, kb0, kb1;
            int slice, parts;
            while (ok && cursor_next(p, cur, tile, slice, kb0, kb1, parts)) {
                if (!mbar_wait(&s->acc_empty[acc], acc_phase ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
                uint32_t first = 0u;      // 0 for the tile's first MMA: overwrite the accumulator
                for (int64_t kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&s->full[stage], phase, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)((stage * C::STAGE_BYTES) >> 4);
                    const uint64_t ad = a_desc0 + so, bd = b_desc0 + so;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_f16(d_tmem, ad + kk * a_step, bd + kk * b_step, idesc, kk > 0 ? 1u : first);
                    first = 1u;
                    mma_commit(&s->empty[stage]);   // stage free once these MMAs finish
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(&s->acc_full[acc]);      // accumulator ready for the epilogue
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            // all MMAs this thread issued have completed once `drain` flips
            mma_commit(&s->drain);
            mbar_wait_drain(&s->drain, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int lane_group = warp & 3;          // TMEM lanes this warp may access
        const int row_in_tile = lane_group * 32 + lane;
        const int etid = threadIdx.x - 64;        // 0..127 across the epilogue warps
        uint32_t acc = 0, acc_phase = 0;
        Cursor cur = cursor_begin(p);
        int64_t tile, kb0, kb1;
        int slice, parts;
        while (cursor_next(p, cur, tile, slice, kb0, kb1, parts)) {
            int64_t item, mb, nb;
            tile_coords(p, tile, item, mb, nb);
            if (!SWAP && (!SPLIT || parts == 1) && mb * BM + row_in_tile < p.M)
                prefetch_residual(p, item, mb * BM + row_in_tile, nb * BN, min64(BN, p.N - nb * BN));
            if (!mbar_wait(&s->acc_full[acc], acc_phase, abort_flag, p.err)) break;
            tc_fence_after();
            const int64_t row = mb * BM + row_in_tile;
            const int64_t rows_total = SWAP ? p.N : p.M;    // extent of the TMEM-lane dimension
            const bool row_ok = row < rows_total;
            const uint32_t t_base =
                tmem_base + ((uint32_t)(lane_group * 32) << 16) + acc * C::ACC_COLS;
            // the whole tile in this piece: narrow and store straight from TMEM
            auto store_direct = [&]() {
                if constexpr (SWAP) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x16(t_base, r);
                    if (row_ok) {
                        unsigned short* y = static_cast<unsigned short*>(p.Y);
#pragma unroll
                        for (int m = 0; m < BN; ++m)
                            if (m < p.M) {
                                unsigned short* yp = y + (item * p.M + m) * p.N + row;
                                *yp = (unsigned short)(pack2(tc_epi(p, __uint_as_float(r[m]), m, row,
                                                                    resid16(p, yp)),
                                                             0.f, p.is_bf16) &
                                                       0xFFFFu);
                            }
                    }
                } else {
                    unsigned char* yrow = static_cast<unsigned char*>(p.Y) +
                                          ((item * p.M + (row_ok ? row : 0)) * p.N) * 2;
#pragma unroll 1
                    for (int c = 0; c < BN; c += CH) {
                        uint32_t r[32];
                        if (CH == 32) tmem_ld_32x32b_x32(t_base + c, r);
                        else tmem_ld_32x32b_x16(t_base + c, r);
                        const int64_t col = nb * BN + c;
                        if constexpr (CH == 32 && !SPLIT) {
                            if (row_ok && col < p.N && p.y_unaligned) {
                                const int valid = (int)min64(32, p.N - col);
                                uint32_t packed[16];
                                epi_run<16>(p, r, row, col, yrow + col * 2, valid, packed);
                                store_run_unaligned(yrow + col * 2, packed, valid);
                                continue;
                            }
                        }
                        if (row_ok && col < p.N) {
                            uint4* dst = reinterpret_cast<uint4*>(yrow + col * 2);
                            // N is a multiple of 8: whole 16-byte groups only
                            const int64_t left = (p.N - col) / 8;
                            const int groups = (int)(left < CH / 8 ? left : CH / 8);
                            uint32_t packed[16];
                            epi_run<CH / 2>(p, r, row, col, yrow + col * 2, groups, packed);
#pragma unroll
                            for (int q = 0; q < CH / 8; ++q)
                                if (q < groups)
                                    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                        packed[4 * q + 2], packed[4 * q + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s->acc_empty[acc]);
            };
            if (!SPLIT || parts == 1) {
                store_direct();
            } else {
                // float32 partial tile of this slice -> part1[tile][slice]
                float* mine = p.part1 + ((tile * p.splits + slice) * BM) * (int64_t)BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += CH) {
                    uint32_t r[32];
                    if (CH == 32) tmem_ld_32x32b_x32(t_base + c, r);
                    else tmem_ld_32x32b_x16(t_base + c, r);
                    if (row_ok) {
                        float4* dst = reinterpret_cast<float4*>(mine + (int64_t)row_in_tile * BN + c);
#pragma unroll
                        for (int q = 0; q < CH / 4; ++q)
                            dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                 __uint_as_float(r[4 * q + 2]),
                                                 __uint_as_float(r[4 * q + 3]));
                    }
                }
                // the accumulator can be refilled while the reduction runs
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s->acc_empty[acc]);

                // fixed two-level reduction tree: slices of one group summed
                // in slice order by the group's last arrival, then the group
                // sums in group order by the last group
                // stream-K: one group holding the tile's contributors
                const int g = p.stream ? 0 : slice / p.group;
                const int gsize = p.stream ? parts : min(p.group, p.splits - g * p.group);
                const int64_t rows_valid = min64(BM, rows_total - mb * BM);
                const int64_t e4_count = rows_valid * BN / 4;
                const int64_t tile_floats = (int64_t)BM * BN;
                __threadfence();
                epi_sync();
                if (etid == 0) {
                    const unsigned int prev = atomicAdd(p.cnt1 + tile * p.groups + g, 1u);
                    s->last_flag = (prev == (unsigned int)gsize - 1) ? 1 : 0;
                }
                epi_sync();
                const int last1 = s->last_flag;
                epi_sync();
                if (last1) {
                    __threadfence();
                    const float* first = p.part1 + (tile * p.splits + g * p.group) * tile_floats;
                    if (p.groups == 1) {
                        for (int64_t e4 = etid; e4 < e4_count; e4 += 2 * EPI_THREADS) {
                            const int64_t e4b = e4 + EPI_THREADS < e4_count ? e4 + EPI_THREADS : -1;
                            float4 v0, v1;
                            ordered_sum4x2(first, tile_floats, gsize, e4, e4b, v0, v1);
                            store_sum(item, mb, nb, e4, v0);
                            if (e4b >= 0) store_sum(item, mb, nb, e4b, v1);
                        }
                        if (etid == 0) p.cnt1[tile * p.groups + g] = 0u;
                    } else {
                        float* gsum = p.part2 + (tile * p.groups + g) * tile_floats;
                        for (int64_t e4 = etid; e4 < e4_count; e4 += 2 * EPI_THREADS) {
                            const int64_t e4b = e4 + EPI_THREADS < e4_count ? e4 + EPI_THREADS : -1;
                            float4 v0, v1;
                            ordered_sum4x2(first, tile_floats, gsize, e4, e4b, v0, v1);
                            reinterpret_cast<float4*>(gsum)[e4] = v0;
                            if (e4b >= 0) reinterpret_cast<float4*>(gsum)[e4b] = v1;
                        }
                        __threadfence();
                        epi_sync();
                        if (etid == 0) {
                            p.cnt1[tile * p.groups + g] = 0u;
                            const unsigned int prev = atomicAdd(p.cnt2 + tile, 1u);
                            s->last_flag = (prev == (unsigned int)p.groups - 1) ? 1 : 0;
                        }
                        epi_sync();
                        const int last2 = s->last_flag;
                        epi_sync();
                        if (last2) {
                            __threadfence();
                            const float* g0 = p.part2 + tile * p.groups * tile_floats;
                            for (int64_t e4 = etid; e4 < e4_count; e4 += 2 * EPI_THREADS) {
                                const int64_t e4b =
                                    e4 + EPI_THREADS < e4_count ? e4 + EPI_THREADS : -1;
                                float4 v0, v1;
                                ordered_sum4x2(g0, tile_floats, p.groups, e4, e4b, v0, v1);
                                store_sum(item, mb, nb, e4, v0);
                                if (e4b >= 0) store_sum(item, mb, nb, e4b, v1);
                            }
                            if (etid == 0) p.cnt2[tile] = 0u;
                        }
                    }
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// 2-CTA variant (cta_group::2) for large FLOAT16 / BFLOAT16 products.
//
// A cluster of two CTAs on one TPC computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256): CTA rank r stages A rows
// m0 + 128 r .. +127 and B columns n0 + 128 r .. +127 in its own shared
// memory, the leader (rank 0) issues the MMAs that read both CTAs' halves,
// and each CTA's TMEM receives its own 128 rows x 256 columns.  Per SM that
// is 32 KB of operands per 64-deep K block instead of 48 KB, so 6 stages and
// an epilogue staging area fit where the 1-CTA kernel has 4 stages.
//
// Synchronisation: both CTAs' TMA loads complete on the leader's full[s]
// barrier (two arrivals: the leader's A loader and B loader each arm it with
// both CTAs' bytes of their operand); the leader's MMA
// commits multicast to empty[s] and acc_full[b] in both CTAs; both CTAs'
// epilogue warps arrive on the leader's acc_empty[b] (8 arrivals).  Both
// CTAs allocate and free TMEM with .cta_group::2, and meet at a cluster
// barrier before exiting so no remote arrival targets a finished CTA.

namespace pair {

constexpr int A_BYTES = 128 * BK * 2;               // this CTA's 128 rows of A
constexpr int B_BYTES = 128 * BK * 2;               // this CTA's 128 columns of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;      // 32 KiB
// warps: 0 loads A, 1 issues the MMAs, 2-5 run the epilogue, 6 loads B (one
// TMA load per K block and lane keeps each issue loop short)
constexpr int PAIR_THREADS = 224;
// 6 stages and an epilogue staging area where each epilogue warp turns its
// 32 rows x 128 bytes (32 float32 columns, or 64 16-bit ones) into runs of
// whole rows (36 words per row, so that both the row-wise writes and the
// column-wise reads are free of bank conflicts)
constexpr int STAGE_PITCH = 36;                     // 32-bit words per staged row
constexpr int STAGING_BYTES = 4 * 32 * STAGE_PITCH * 4;   // 4 warps: 18 KiB
template <bool F8>
constexpr int stages() { return 6; }
template <bool F8>
constexpr int smem_bytes() {
    return stages<F8>() * STAGE_BYTES + STAGING_BYTES + 1024 + 512;
}
constexpr int TMEM_COLS = 512;                       // two 256-column accumulators

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `local` in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to(const void* local, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
    return out;
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// TMA load into this CTA's shared memory, completing on an mbarrier that may
// be in the peer CTA (shared::cluster address)
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void mma2_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma2_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// kind::f8f6f4 instruction descriptor: float32 accumulator (bits 4-5 = 1), A
// and B formats in bits 7-9 / 10-12 (0 = E4M3, 1 = E5M2), both K-major, N >> 3
// in bits 17-22, M >> 4 in bits 24-28
__host__ __device__ constexpr uint32_t f8_desc(int fmt, int m, int n) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// arrive on the barrier at this offset in both CTAs of the pair once the
// MMAs issued so far have completed
__device__ __forceinline__ void commit2_both(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)), "h"((unsigned short)0x3)
        : "memory");
}

// arrive on this CTA's own barrier once the MMAs issued so far have completed
__device__ __forceinline__ void commit2_local(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// F8: 8-bit float operands, both K-major (B given as [N, K]), 128 elements
// per 128-byte swizzle row and 32 per MMA (kind::f8f6f4), float32 output;
// the byte geometry of the shared-memory stages is the same as for 16-bit
// operands with K-major B.
template <bool F8>
__global__ void __launch_bounds__(PAIR_THREADS, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_b, const Params p) {
    constexpr int STAGES = stages<F8>();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* staging = reinterpret_cast<float*>(base + STAGES * STAGE_BYTES);
    Smem* s = reinterpret_cast<Smem*>(base + STAGES * STAGE_BYTES + STAGING_BYTES);
    volatile int* abort_flag = &s->abort_flag;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // pair tiles: 256 rows x 256 columns, persistent over the clusters
    const int64_t ptm = ceil_div(p.M, 256), ptn = ceil_div(p.N, 256);
    const int64_t per_item = ptm * ptn;
    const int64_t total = per_item * p.items;
    // work units: tiles [0, pair_full) whole, then each later tile as two
    // halves of 128 columns, so that a last partial wave of r tiles keeps
    // 2r clusters busy for half as long
    const int64_t full = total - (p.pair_half_tiles < total ? p.pair_half_tiles : total);
    const int64_t units = full + 2 * (total - full);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s->full[i], 2);        // the leader's A and B loaders arm it
            mbar_init(&s->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s->acc_full[i], 1);
            mbar_init(&s->acc_empty[i], 8);   // 4 epilogue warps in each CTA
        }
        mbar_init(&s->drain, 1);
        s->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc2(&s->tmem_base, TMEM_COLS);
    tc_fence_before();
    cluster_sync();          // both CTAs' barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = s->tmem_base;
    grid_dependency_wait();
    grid_launch_dependents();

    // unit u -> tile and half (-1: the whole 256 columns; 0 / 1: columns
    // 0..127 / 128..255 of the tile)
    auto unit_tile = [&](int64_t u, int& half) -> int64_t {
        if (u < full) {
            half = -1;
            return u;
        }
        half = (int)((u - full) & 1);
        return full + (u - full) / 2;
    };
    auto coords = [&](int64_t t, int64_t& item, int64_t& mb, int64_t& nb) {
        item = t / per_item;
        const int64_t r = t % per_item;
        const int64_t group_span = (int64_t)8 * ptn;      // 8 pair rows per raster group
        const int64_t g = r / group_span;
        const int64_t first = g * 8;
        const int64_t gm = min64(ptm - first, 8);
        const int64_t in = r % group_span;
        mb = first + in % gm;
        nb = in / gm;
    };

    if (warp == 0 || warp == 6) {
        if (lane == 0) {
            // warp 0 loads A, warp 6 loads B, each waiting for the same free
            // stages; the leader's two loaders each arm the leader's full
            // barrier with their operand's bytes from both CTAs.  The issue
            // loop is on the critical path (one K block every 512 MMA
            // cycles): shared and cluster addresses advance by adds, and the
            // stages armed for the abort drain are bits in registers
            const bool load_a = warp == 0;
            if (load_a)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            else
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            const uint32_t stage0 = smem_u32(base);
            const uint32_t full0_leader = map_to(&s->full[0], 0);
            const uint32_t a_tma_bytes = p.a_mn ? 64 * BK * 2 : 0;     // second A box, if any
            uint32_t stage = 0, phase = 0, armed_bits = 0, parity_bits = 0;
            bool ok = true;
            for (int64_t u = cluster_id(); u < units && ok; u += cluster_count()) {
                int half;
                const int64_t t = unit_tile(u, half);
                int64_t item, mb, nb;
                coords(t, item, mb, nb);
                int64_t a_off, b_off;
                batch_offsets(p.map, item, a_off, b_off);
                const int a_item = (int)(a_off / p.a_item_elems);
                const int b_item = (int)(b_off / p.b_item_elems);
                // each CTA stages its half of the unit's B columns: 128 of a
                // whole tile, 64 of a half tile
                const int m0 = (int)(mb * 256 + rank * 128);
                const int n0 = half < 0 ? (int)(nb * 256 + rank * 128) : (int)(nb * 256 + half * 128 + rank * 64);
                // this loader's bytes landing on the leader's full barrier
                // from both CTAs; the 4-D B load brings two 64-column blocks
                // for half tiles too (the second one unused)
                const uint32_t tx = load_a ? 2u * A_BYTES : ((half < 0 || p.b_blocks) ? 2u * B_BYTES : B_BYTES);
                const int k_step = F8 ? 128 : BK;
                int k0 = 0;
                for (int64_t kb = 0; kb < p.k_blocks; ++kb, k0 += k_step) {
                    if (!mbar_wait(&s->empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    const uint32_t sa = stage0 + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t full_leader = full0_leader + stage * (uint32_t)sizeof(uint64_t);
                    if (leader) {
                        mbar_arrive_expect_tx(&s->full[stage], tx);
                        armed_bits |= 1u << stage;
                        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    }
                    if (load_a) {
                        if (!a_tma_bytes) {
                            tma_load_3d_pair(sa, &tmap_a, full_leader, k0, m0, a_item);
                        } else {
                            tma_load_3d_pair(sa, &tmap_a, full_leader, m0, k0, a_item);
                            tma_load_3d_pair(sa + a_tma_bytes, &tmap_a, full_leader, m0 + 64, k0, a_item);
                        }
                    } else if (p.b_blocks) {
                        tma_load_4d_pair(sb, &tmap_b, full_leader, 0, k0, n0 >> 6, b_item);
                    } else if (!p.b_k) {
                        tma_load_3d_pair(sb, &tmap_b, full_leader, n0, k0, b_item);
                        if (half < 0)
                            tma_load_3d_pair(sb + 64 * BK * 2, &tmap_b, full_leader, n0 + 64, k0, b_item);
                    } else {
                        tma_load_3d_pair(sb, &tmap_b, full_leader, k0, n0, b_item);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (*abort_flag && leader) {
                for (int i = 0; i < STAGES; ++i)
                    if ((armed_bits >> i) & 1u) mbar_wait_drain(&s->full[i], (parity_bits >> i) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = F8 ? f8_desc(p.f8_fmt, 256, 256)
                                      : instr_desc(p.is_bf16, 256, 256, p.a_mn, p.b_k ? 0 : 1);
            const uint32_t idesc_half = F8 ? idesc : instr_desc(p.is_bf16, 256, 128, p.a_mn, p.b_k ? 0 : 1);
            // descriptors of stage 0, built once: a later stage and each
            // 16-deep step add their byte offset >> 4 to the start-address
            // field (bits 0-13), which no shared-memory address overflows.
            // Issuing one K block must take well under the 512 cycles its
            // four MMAs run for.
            const uint32_t stage0 = smem_u32(base);
            const uint64_t a_desc0 = p.a_mn ? smem_desc(stage0, 64 * BK * 2, 1024, 2u)
                                            : smem_desc(stage0, 16, 1024, 2u);
            const uint64_t b_desc0 = p.b_k ? smem_desc(stage0 + A_BYTES, 16, 1024, 2u)
                                           : smem_desc(stage0 + A_BYTES, 64 * BK * 2, 1024, 2u);
            const uint64_t a_step = p.a_mn ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
            const uint64_t b_step = p.b_k ? (UMMA_K * 2) >> 4 : (UMMA_K * 128) >> 4;
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t u = cluster_id(); u < units && ok; u += cluster_count()) {
                int half;
                unit_tile(u, half);
                const uint32_t id = half < 0 ? idesc : idesc_half;
                if (!mbar_wait(&s->acc_empty[acc], acc_phase ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * 256;
                uint32_t first = 0u;      // 0 for the unit's first MMA: overwrite the accumulator
                for (int64_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&s->full[stage], phase, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
                    const uint64_t ad = a_desc0 + so, bd = b_desc0 + so;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        if constexpr (F8) mma2_f8(d_tmem, ad + kk * a_step, bd + kk * b_step, id, kk > 0 ? 1u : first);
                        else mma2_f16(d_tmem, ad + kk * a_step, bd + kk * b_step, id, kk > 0 ? 1u : first);
                    }
                    first = 1u;
                    commit2_both(&s->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                commit2_both(&s->acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            commit2_local(&s->drain);
            mbar_wait_drain(&s->drain, 0);
        }
    } else {
        const int lane_group = warp & 3;
        const int row_in_tile = lane_group * 32 + lane;
        const uint32_t acc_empty_leader[2] = {map_to(&s->acc_empty[0], 0), map_to(&s->acc_empty[1], 0)};
        uint32_t acc = 0, acc_phase = 0;
        for (int64_t u = cluster_id(); u < units; u += cluster_count()) {
            int half;
            const int64_t t = unit_tile(u, half);
            int64_t item, mb, nb;
            coords(t, item, mb, nb);
            // the unit's columns: [cbase, cbase + width) of the output
            const int64_t cbase = nb * 256 + (half < 0 ? 0 : half * 128);
            const int width = half < 0 ? 256 : 128;
            if (!F8 && mb * 256 + rank * 128 + row_in_tile < p.M)
                prefetch_residual(p, item, mb * 256 + rank * 128 + row_in_tile, cbase,
                                  min64(width, p.N - cbase));
            if (!mbar_wait(&s->acc_full[acc], acc_phase, abort_flag, p.err)) break;
            tc_fence_after();
            const int64_t row = mb * 256 + rank * 128 + row_in_tile;
            const bool row_ok = row < p.M;
            const uint32_t t_base = tmem_base + ((uint32_t)(lane_group * 32) << 16) + acc * 256;
            if constexpr (F8) {
                // float32 output rows; N is a multiple of 4: whole 16-byte
                // groups.  Each 32-column run goes through this warp's
                // staging rows, so that a warp store writes 4 rows x 128
                // bytes instead of 16 bytes in each of 32 rows
                float* yrow = static_cast<float*>(p.Y) + (item * p.M + (row_ok ? row : 0)) * p.N;
                float* stage_rows = staging + lane_group * 32 * STAGE_PITCH;
                const int64_t row0 = mb * 256 + rank * 128 + lane_group * 32;   // the warp's first row
                const int cq = lane & 7;                  // 16-byte group this lane writes back
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_base + c, r);
                    const int64_t col = nb * 256 + c;
                    if (col >= p.N) continue;             // warp-uniform: the whole run is past N
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    if (p.epi.mode != 0 && row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col + i < p.N)
                                v[i] = apply_epilogue<float>(p.epi, v[i], row, col + i, yrow + col + i);
                    }
                    float4* mine = reinterpret_cast<float4*>(stage_rows + lane * STAGE_PITCH);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mine[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    __syncwarp();
                    const int64_t gcol = col + cq * 4;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int rr = (lane >> 3) + 4 * j;
                        const int64_t grow = row0 + rr;
                        const float4 w = *reinterpret_cast<const float4*>(stage_rows + rr * STAGE_PITCH + cq * 4);
                        if (grow < p.M && gcol < p.N)
                            *reinterpret_cast<float4*>(static_cast<float*>(p.Y) + (item * p.M + grow) * p.N + gcol) = w;
                    }
                    __syncwarp();                          // the rows are rewritten by the next run
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) remote_arrive(acc_empty_leader[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                continue;
            }
            unsigned char* yrow = static_cast<unsigned char*>(p.Y) +
                                  ((item * p.M + (row_ok ? row : 0)) * p.N) * 2;
            if (!p.y_unaligned) {
                // 64-column runs (two TMEM loads) through this warp's staging
                // rows, so that a warp store writes 4 rows x 128 bytes; Y's
                // rows are 16-byte multiples here (N % 8 == 0)
                uint32_t* stage_rows = reinterpret_cast<uint32_t*>(staging) + lane_group * 32 * STAGE_PITCH;
                const int64_t row0 = mb * 256 + rank * 128 + lane_group * 32;   // the warp's first row
                const int cq = lane & 7;                  // 16-byte group this lane writes back
#pragma unroll 1
                for (int c = 0; c < width; c += 64) {
                    uint32_t packed[32];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(t_base + c + hh * 32, r);
                        const int64_t col = cbase + c + hh * 32;
                        if (row_ok && col < p.N) {
                            const int64_t left = (p.N - col) / 8;
                            const int groups = (int)(left < 4 ? left : 4);
                            epi_run<16>(p, r, row, col, yrow + col * 2, groups, packed + hh * 16);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) packed[hh * 16 + i] = 0u;   // never stored
                        }
                    }
                    const int64_t col0 = cbase + c;
                    if (col0 >= p.N) continue;            // warp-uniform: the whole run is past N
                    uint4* mine = reinterpret_cast<uint4*>(stage_rows + lane * STAGE_PITCH);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mine[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    __syncwarp();
                    const int64_t gcol = col0 + cq * 8;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int rr = (lane >> 3) + 4 * j;
                        const int64_t grow = row0 + rr;
                        const uint4 w = *reinterpret_cast<const uint4*>(stage_rows + rr * STAGE_PITCH + cq * 4);
                        if (grow < p.M && gcol < p.N)
                            *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.Y) +
                                                      ((item * p.M + grow) * p.N + gcol) * 2) = w;
                    }
                    __syncwarp();                          // the rows are rewritten by the next run
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) remote_arrive(acc_empty_leader[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < width; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c, r);
                const int64_t col = cbase + c;
                if (row_ok && col < p.N && p.y_unaligned) {
                    const int valid = (int)min64(32, p.N - col);
                    uint32_t packed[16];
                    epi_run<16>(p, r, row, col, yrow + col * 2, valid, packed);
                    store_run_unaligned(yrow + col * 2, packed, valid);
                } else if (row_ok && col < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + col * 2);
                    const int64_t left = (p.N - col) / 8;
                    const int groups = (int)(left < 4 ? left : 4);
                    uint32_t packed[16];
                    epi_run<16>(p, r, row, col, yrow + col * 2, groups, packed);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < groups)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                                packed[4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) remote_arrive(acc_empty_leader[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();          // no remote arrival may target a CTA that has left
    tc_fence_after();
    if (warp == 1) tmem_dealloc2(tmem_base, TMEM_COLS);
}

}  // namespace pair

// ---------------------------------------------------------------------------
// Split-K for tiny outputs (M <= 32, N <= 32, FP16/BF16).
//
// A 128-row tcgen05 MMA would leave 3/4 of its rows idle here and its cost
// per instruction does not shrink with N, so this kernel keeps the TMA
// staging but multiplies with warp-level mma.sync.m16n8k16 (float32
// accumulation): CTA s owns K slice s, one producer lane streams the
// slice's 64-deep chunks (A: 32 rows x 128 bytes, 128-byte swizzle; B: 64
// K-rows x 64 bytes, 64-byte swizzle) through a ring of full/empty
// mbarriers, and four MMA warps each take one 16-deep step of every chunk
// (ldmatrix on the swizzled layouts, ldmatrix.trans for B).  The four warps'
// 32 x 32 sums are added in warp order, and the slices are reduced by the
// same fixed two-level tree as the tensor-core split-K (slices of a group in
// order by the group's last arrival, then the groups in order).

namespace tiny {

// Split-K for outputs of at most 32 x 32: one K slice per CTA, CTAs in
// clusters of CL.  Each CTA's 32 x 32 partial stays in its shared memory; CTA
// r of a cluster sums rows [r * 32 / CL, (r + 1) * 32 / CL) of the CL partials
// through distributed shared memory and writes that cluster sum; the last
// cluster to deliver a row band sums the cluster sums in cluster order and
// stores.  Every sum runs in a fixed order, so the result is the same run to
// run.
constexpr int ROWS = 32, COLS = 32;
constexpr int A_CHUNK = ROWS * BK * 2;             // 4 KiB
constexpr int B_CHUNK = BK * COLS * 2;             // 4 KiB
constexpr int CHUNK = A_CHUNK + B_CHUNK;
constexpr int STAGES = 24;
constexpr int MMA_WARPS = 4;
constexpr int MMA_THREADS = MMA_WARPS * 32;
constexpr int THREADS_T = (MMA_WARPS + 1) * 32;    // + one producer warp
constexpr int RED_BYTES = MMA_WARPS * ROWS * (COLS + 1) * 4;
constexpr int TILE_BYTES = ROWS * COLS * 4;        // this CTA's partial (float32)
constexpr int SMEM_BYTES = STAGES * CHUNK + RED_BYTES + TILE_BYTES + 1024 + 512;
constexpr int LOAD_BATCH = 8;                      // cluster sums loaded per round trip

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    int abort_flag;
    int last_flag;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, int is_bf16) {
    if (is_bf16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cluster4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
// arrival count with release (this CTA's earlier writes, ordered before it by
// a block barrier) and acquire (the other arrivals' writes) at GPU scope
__device__ __forceinline__ unsigned int arrive_acq_rel(unsigned int* counter) {
    unsigned int prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
    return prev;
}

template <int CL>
__global__ void __launch_bounds__(THREADS_T, 1)
splitk_tiny_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const Params p) {
    static_assert(CL == 2 || CL == 4 || CL == 8, "cluster of 2, 4 or 8 CTAs");
    constexpr int BAND_ROWS = ROWS / CL;                 // rows this CTA reduces
    constexpr int BAND_F4 = BAND_ROWS * COLS / 4;        // float4s of one band
    constexpr int PARTS = MMA_THREADS / BAND_F4;         // threads per float4 at level 2
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* red = reinterpret_cast<float*>(base + STAGES * CHUNK);           // [4][32][33]
    float* tile = reinterpret_cast<float*>(base + STAGES * CHUNK + RED_BYTES);   // [32][32]
    Bars* s = reinterpret_cast<Bars*>(base + STAGES * CHUNK + RED_BYTES + TILE_BYTES);
    volatile int* abort_flag = &s->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const int slice = blockIdx.x;
    const int rank = (int)pair::cluster_rank();
    const int cluster = slice / CL;
    // K blocks split evenly: slice s takes [s * kb / S, (s + 1) * kb / S)
    const int64_t kb0 = (int64_t)slice * p.k_blocks / p.splits;
    const int64_t kb1 = (int64_t)(slice + 1) * p.k_blocks / p.splits;
    const int nchunks = kb1 > kb0 ? (int)(kb1 - kb0) : 0;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->empty[i], MMA_WARPS);
        }
        s->abort_flag = 0;
        s->last_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // nothing global is read or written before the previous grid is done
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == MMA_WARPS) {
        // producer: one lane issues every chunk's two TMA loads
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            uint32_t armed_parity[STAGES];
            bool armed[STAGES];
            for (int i = 0; i < STAGES; ++i) armed[i] = false;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % STAGES;
                const uint32_t ph = (uint32_t)(c / STAGES) & 1u;
                if (!mbar_wait(&s->empty[st], ph ^ 1, abort_flag, p.err)) break;
                unsigned char* sa = base + st * CHUNK;
                mbar_arrive_expect_tx(&s->full[st], CHUNK);
                armed[st] = true;
                armed_parity[st] = ph;
                const int k0 = (int)((kb0 + c) * BK);
                tma_load_3d(sa, &tmap_a, &s->full[st], k0, 0, 0);
                tma_load_3d(sa + A_CHUNK, &tmap_b, &s->full[st], 0, k0, 0);
            }
            if (*abort_flag)
                for (int i = 0; i < STAGES; ++i)
                    if (armed[i]) mbar_wait_drain(&s->full[i], armed_parity[i]);
        }
        __syncwarp();
    } else {
        // MMA warps: warp w takes the 16-deep step w of every chunk
        float acc[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;
        const int q = lane >> 3, r8 = lane & 7;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % STAGES;
            const uint32_t ph = (uint32_t)(c / STAGES) & 1u;
            if (!mbar_wait(&s->full[st], ph, abort_flag, p.err)) break;
            const uint32_t a_base = smem_u32(base + st * CHUNK);
            const uint32_t b_base = a_base + A_CHUNK;
            uint32_t a[2][4], b[2][4];
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
                // rows mb*16 + (q&1)*8 + r8, 16-byte chunk 2*warp + (q>>1); 128-byte swizzle
                const int r = mb * 16 + (q & 1) * 8 + r8;
                const int kc = warp * 2 + (q >> 1);
                ldsm_x4(a_base + r * 128 + ((kc ^ (r & 7)) << 4), a[mb]);
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                // K rows warp*16 + (q&1)*8 + r8, 16-byte chunk 2*np + (q>>1); 64-byte swizzle
                const int kr = warp * 16 + (q & 1) * 8 + r8;
                const int nc = np * 2 + (q >> 1);
                ldsm_x4_t(b_base + kr * 64 + ((nc ^ ((kr >> 1) & 3)) << 4), b[np]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s->empty[st]);
#pragma unroll
            for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                for (int nb = 0; nb < 4; ++nb)
                    mma16816(acc[mb][nb], a[mb], b[nb >> 1][(nb & 1) * 2], b[nb >> 1][(nb & 1) * 2 + 1],
                             p.is_bf16);
        }
        // this warp's 32 x 32 sums -> red[warp]
        float* mine = red + warp * ROWS * (COLS + 1);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                const int row = mb * 16 + (lane >> 2), col = nb * 8 + 2 * (lane & 3);
                mine[row * (COLS + 1) + col] = acc[mb][nb][0];
                mine[row * (COLS + 1) + col + 1] = acc[mb][nb][1];
                mine[(row + 8) * (COLS + 1) + col] = acc[mb][nb][2];
                mine[(row + 8) * (COLS + 1) + col + 1] = acc[mb][nb][3];
            }
        epi_sync();
        // the slice's partial: warp sums in warp order -> tile
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int idx = tid + e * MMA_THREADS;
            const int row = idx / COLS, col = idx % COLS;
            float v = red[row * (COLS + 1) + col];
#pragma unroll
            for (int w = 1; w < MMA_WARPS; ++w) v += red[w * ROWS * (COLS + 1) + row * (COLS + 1) + col];
            tile[idx] = v;
        }
    }
    // every CTA of the cluster holds its partial
    cluster_arrive();
    cluster_wait();

    // level 1: this CTA's row band summed over the cluster's CTAs in rank
    // order, through distributed shared memory
    const int band0 = rank * BAND_ROWS * COLS;            // first float of the band
    if (tid < BAND_F4) {
        float4 x[CL];
#pragma unroll
        for (int r = 0; r < CL; ++r) x[r] = ld_cluster4(pair::map_to(tile + band0 + tid * 4, r));
        float4 v = x[0];
#pragma unroll
        for (int r = 1; r < CL; ++r) add4(v, x[r]);
        reinterpret_cast<float4*>(p.part1 + (int64_t)cluster * ROWS * COLS + band0)[tid] = v;
    }
    // done with the other CTAs' shared memory (waited for before exit)
    cluster_arrive();

    // level 2: the last cluster to deliver this band sums the cluster sums
    __syncthreads();
    if (tid == 0) {
        const unsigned int prev = arrive_acq_rel(p.cnt1 + rank);
        s->last_flag = (prev == (unsigned int)p.groups - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s->last_flag && tid < MMA_THREADS) {
        const int f = tid % BAND_F4, part = tid / BAND_F4;
        const int c0 = part * p.groups / PARTS, c1 = (part + 1) * p.groups / PARTS;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4* src = reinterpret_cast<const float4*>(p.part1 + band0) + f;
        for (int cb = c0; cb < c1; cb += LOAD_BATCH) {
            float4 x[LOAD_BATCH];
#pragma unroll
            for (int j = 0; j < LOAD_BATCH; ++j)
                if (cb + j < c1) x[j] = __ldcg(src + (int64_t)(cb + j) * (ROWS * COLS / 4));
#pragma unroll
            for (int j = 0; j < LOAD_BATCH; ++j)
                if (cb + j < c1) add4(v, x[j]);
        }
        // the parts' sums in part order (red is free again)
        float4* parts = reinterpret_cast<float4*>(red);
        parts[part * BAND_F4 + f] = v;
        epi_sync();
        if (part == 0) {
            float4 t = parts[f];
#pragma unroll
            for (int q2 = 1; q2 < PARTS; ++q2) add4(t, parts[q2 * BAND_F4 + f]);
            const int e = band0 + f * 4;
            const int row = e / COLS, col = e % COLS;
            if (row < p.M && col < p.N) store4(p, 0, row, col, t);
        }
        if (tid == 0) p.cnt1[rank] = 0u;
    }
    // no CTA leaves while another may still read its partial
    cluster_wait();
}

}  // namespace tiny

// ---------------------------------------------------------------------------
// Cluster split-K for general FP16/BF16 products whose 128 x 256 tiles leave
// most SMs idle (a few hundred rows, or a narrow N): the K blocks of each
// tile are cut into `ways` slices, one per CTA of a thread-block cluster.
// Each CTA streams its slice of A and B through a 4-stage TMA ring into a
// 128 x 256 TMEM accumulator, stages the accumulator as a float32 partial
// tile in its own shared memory (the ring, idle by then) and copies its
// valid rows, in coalesced 16-byte groups, to its slot of a plan-owned
// workspace (L2-resident).  After one cluster barrier each CTA sums a
// contiguous band of the tile's 8-column runs over the cluster's partials,
// read from L2 in slice order (so the result does not depend on timing),
// runs the epilogue and stores.  No atomics.

namespace csplit {

constexpr int BN = 256;
constexpr int A_BYTES = BM * BK * 2;               // 16 KiB (rows past M: stale, never stored)
constexpr int B_BYTES = BK * BN * 2;               // 32 KiB: four 64-column MN-major blocks
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // 48 KiB
constexpr int STAGES = 4;
constexpr int PART_PITCH = BN + 4;                 // floats per partial row: float4 rows 16 B apart in banks
constexpr int PART_BYTES = BM * PART_PITCH * 4;    // 133,120 bytes, inside the idle ring
static_assert(PART_BYTES <= STAGES * STAGE_BYTES, "the partial tile fits in the ring");
constexpr int THREADS_CS = 192;                    // producer, MMA issuer, 4 epilogue warps
constexpr int TMEM_COLS = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int MAX_WAYS = 8;

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    int abort_flag;
    uint32_t tmem_base;
};

__global__ void __launch_bounds__(THREADS_CS, 1)
csplit_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
              const Params p, int ways, int64_t kb_per) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* s = reinterpret_cast<Bars*>(base + STAGES * STAGE_BYTES);
    float* part = reinterpret_cast<float*>(base);          // after the main loop
    volatile int* abort_flag = &s->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = (int)pair::cluster_rank();            // this CTA's K slice
    const int64_t tile = pair::cluster_id();
    const int64_t item = tile / p.tiles_per_item;
    const int64_t r_in = tile % p.tiles_per_item;
    const int64_t mb = r_in / p.tiles_n, nb = r_in % p.tiles_n;
    const int64_t kb0 = rank * kb_per;
    const int64_t kb1 = min64(p.k_blocks, kb0 + kb_per);   // the host leaves no slice empty

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->empty[i], 1);
        }
        mbar_init(&s->acc_full, 1);
        s->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(&s->tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s->tmem_base;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0 && lane == 0) {
        // ---- producer
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
        int64_t a_off, b_off;
        batch_offsets(p.map, item, a_off, b_off);
        const int a_item = (int)(a_off / p.a_item_elems);
        const int b_item = (int)(b_off / p.b_item_elems);
        const int m0 = (int)(mb * BM), n0 = (int)(nb * BN);
        const uint32_t stage0 = smem_u32(base);
        const uint32_t full0 = smem_u32(&s->full[0]);
        uint32_t stage = 0, phase = 0, armed_bits = 0, parity_bits = 0;
        int k0 = (int)(kb0 * BK);
        for (int64_t kb = kb0; kb < kb1; ++kb, k0 += BK) {
            if (!mbar_wait(&s->empty[stage], phase ^ 1, abort_flag, p.err)) break;
            const uint32_t sa = stage0 + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            const uint32_t fb = full0 + stage * (uint32_t)sizeof(uint64_t);
            mbar_arrive_expect_tx(&s->full[stage], p.stage_tx_bytes);
            armed_bits |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            tma_load_3d(sa, &tmap_a, fb, k0, m0, a_item);
            if (p.b_blocks) {
                asm volatile(
                    "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(sb),
                    "l"(reinterpret_cast<uint64_t>(&tmap_b)), "r"(fb), "r"(0), "r"(k0), "r"(n0 >> 6),
                    "r"(b_item)
                    : "memory");
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tma_load_3d(sb + j * (BK * 128), &tmap_b, fb, n0 + 64 * j, k0, b_item);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (*abort_flag) {
            for (int i = 0; i < STAGES; ++i)
                if ((armed_bits >> i) & 1u) mbar_wait_drain(&s->full[i], (parity_bits >> i) & 1u);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: A K-major (128-byte swizzle, 32 bytes per 16-deep
        // step), B MN-major (64-column blocks 8 KiB apart, 16 K-rows of 128
        // bytes per step); descriptors advanced by adds
        const uint32_t idesc = instr_desc(p.is_bf16, BM, BN, 0, 1);
        const uint32_t stage0 = smem_u32(base);
        const uint64_t a_desc0 = smem_desc(stage0, 16, 1024, 2u);
        const uint64_t b_desc0 = smem_desc(stage0 + A_BYTES, BK * 128, 1024, 2u);
        uint32_t stage = 0, phase = 0, first = 0u;
        for (int64_t kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&s->full[stage], phase, abort_flag, p.err)) break;
            tc_fence_after();
            const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
                mma_f16(tmem_base, a_desc0 + so + kk * 2, b_desc0 + so + kk * 128, idesc, kk > 0 ? 1u : first);
            first = 1u;
            mma_commit(&s->empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        mma_commit(&s->acc_full);      // every MMA issued above has completed once it flips
    } else if (warp >= 2) {
        // ---- accumulator -> this CTA's float32 partial tile (all 128 rows;
        // the rows past M are never read back)
        const int lane_group = warp & 3;
        const int row_in_tile = lane_group * 32 + lane;
        if (mbar_wait(&s->acc_full, 0, abort_flag, p.err)) {
            tc_fence_after();
            const uint32_t t_base = tmem_base + ((uint32_t)(lane_group * 32) << 16);
            float4* prow = reinterpret_cast<float4*>(part + row_in_tile * PART_PITCH);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c, r);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    prow[c / 4 + q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                  __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // the valid rows of the partial tile to the plan's workspace (rows of
    // 256 floats; consecutive threads write consecutive 16-byte groups)
    const int64_t rows_valid = min64(BM, p.M - mb * BM);
    float* mine = p.part1 + (tile * ways + rank) * (int64_t)(BM * BN);
    for (int64_t e = threadIdx.x; e < rows_valid * (BN / 4); e += THREADS_CS) {
        const int row = (int)(e / (BN / 4)), c4 = (int)(e % (BN / 4));
        reinterpret_cast<float4*>(mine + (int64_t)row * BN)[c4] =
            reinterpret_cast<const float4*>(part + row * PART_PITCH)[c4];
    }
    pair::cluster_sync();              // every CTA's partial tile is in the workspace (cluster scope)

    // ---- this CTA's share of the tile: a contiguous band of its 8-column
    // runs (runs [rank * runs / ways, (rank + 1) * runs / ways)) over the
    // valid rows, summed over the slices in slice order from L2
    {
        const int64_t cols_valid = min64(BN, p.N - nb * BN);
        const int runs = (int)ceil_div(cols_valid, 8);
        const int run0 = rank * runs / ways, run1 = (rank + 1) * runs / ways;
        const int my_runs = run1 - run0;
        const int64_t items = my_runs > 0 ? rows_valid * my_runs : 0;
        const float* first = p.part1 + tile * ways * (int64_t)(BM * BN);
        for (int64_t e = threadIdx.x; e < items; e += THREADS_CS) {
            const int row = (int)(e / my_runs);
            const int run = run0 + (int)(e % my_runs);
            const float* src = first + (int64_t)row * BN + run * 8;
            float4 x0[MAX_WAYS], x1[MAX_WAYS];
#pragma unroll
            for (int j = 0; j < MAX_WAYS; ++j) {
                if (j < ways) {
                    x0[j] = __ldcg(reinterpret_cast<const float4*>(src + (int64_t)j * BM * BN));
                    x1[j] = __ldcg(reinterpret_cast<const float4*>(src + (int64_t)j * BM * BN + 4));
                }
            }
            float4 a0 = x0[0], a1 = x1[0];
#pragma unroll
            for (int j = 1; j < MAX_WAYS; ++j) {
                if (j < ways) {
                    a0.x += x0[j].x; a0.y += x0[j].y; a0.z += x0[j].z; a0.w += x0[j].w;
                    a1.x += x1[j].x; a1.y += x1[j].y; a1.z += x1[j].z; a1.w += x1[j].w;
                }
            }
            const int64_t grow = mb * BM + row;
            const int64_t gcol = nb * BN + run * 8;
            unsigned char* dst = static_cast<unsigned char*>(p.Y) + ((item * p.M + grow) * p.N + gcol) * 2;
            const uint32_t r8[8] = {__float_as_uint(a0.x), __float_as_uint(a0.y), __float_as_uint(a0.z),
                                    __float_as_uint(a0.w), __float_as_uint(a1.x), __float_as_uint(a1.y),
                                    __float_as_uint(a1.z), __float_as_uint(a1.w)};
            uint32_t packed[4];
            epi_run<4>(p, r8, grow, gcol, dst, 1, packed);
            *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace csplit

// ---------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        cudaGetLastError();
    });
    return fn;
}

// rank-3 map over [items][rows][cols] (cols innermost), 16-bit elements,
// rows `ld` elements apart (0: dense, ld = cols), box {box_cols, box_rows, 1}
// with the given swizzle
static bool encode_3d(CUtensorMap* map, const void* base, int is_bf16, uint64_t cols,
                      uint64_t rows, uint64_t items, uint32_t box_cols, uint32_t box_rows,
                      CUtensorMapSwizzle swizzle, uint64_t ld = 0) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (ld == 0) ld = cols;
    cuuint64_t dims[3] = {cols, rows, items};
    cuuint64_t strides[2] = {ld * 2, ld * rows * 2};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// rank-4 view of a row-major [items][K][N] 16-bit B (rows `ld` elements
// apart, N a multiple of 64) as [items][N / 64][K][64]: a box {64, BK,
// blocks, 1} is `blocks` 64-column MN-major blocks of BK rows, one after the
// other in shared memory (the layout of 3-D boxes at n0, n0 + 64, ...), in
// one TMA load
static bool encode_b_blocks(CUtensorMap* map, const void* base, int is_bf16, uint64_t n, uint64_t k,
                            uint64_t items, uint64_t ld, uint32_t blocks = 2) {
    auto fn = encode_fn();
    if (!fn || n % 64 != 0) return false;
    cuuint64_t dims[4] = {64, k, n / 64, items};
    cuuint64_t strides[3] = {ld * 2, 128, ld * k * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)BK, blocks, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN>
static CUtensorMapSwizzle b_swizzle() {
    return Cfg<BN>::SW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : (Cfg<BN>::SW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B);
}

// The general tiles' operand requirements: 16-bit types, coordinates in
// int32, 16-byte aligned A and B with 16-byte row pitches (TMA), and a dense
// or aligned Y unless the launch stores Y by alignment (y_unaligned).
static bool tc_operands_ok(olc_dtype dt, const Problem& pr, int64_t a_ld, int64_t b_ld) {
    if (dt != OLC_FLOAT16 && dt != OLC_BFLOAT16) return false;
    if (pr.M >= (1LL << 31) || pr.N >= (1LL << 31) || pr.K >= (1LL << 31)) return false;
    if ((reinterpret_cast<uintptr_t>(pr.A) & 15) || (reinterpret_cast<uintptr_t>(pr.B) & 15))
        return false;
    // stored row lengths: A [M, K] or [K, M] (transA), B [K, N] or [N, K] (transB)
    if (pr.a_trans ? (pr.M % 8 != 0 || pr.a_ld) : (a_ld % 8 != 0 || a_ld < pr.K)) return false;
    if (pr.b_trans ? (pr.K % 8 != 0 || pr.b_ld) : (b_ld % 8 != 0 || b_ld < pr.N)) return false;
    if (!pr.y_unaligned && ((reinterpret_cast<uintptr_t>(pr.Y) & 15) || pr.N % 8 != 0)) return false;
    return true;
}

// Shape of a split-K launch: slices, group size, workspace layout.
struct SplitPlan {
    int splits = 1, group = 1, groups = 1;
    int64_t kb_per_split = 0;
    int64_t tiles = 0;
    size_t part1_bytes = 0, part2_bytes = 0, counters = 0;
    bool stream = false;       // stream-K shares instead of equal slices
    int64_t grid = 0;          // stream-K: CTAs (one share each)
};

// Stream-K: `grid` CTAs share the tiles' K blocks equally; a tile cut
// between CTAs has at most `splits` contributors, summed in K order by the
// last one (one load batch, so at most SUM_BATCH contributors).
template <int BN>
static SplitPlan stream_plan(int64_t tiles, int64_t k_blocks, int sm_count) {
    SplitPlan sp;
    const int64_t iters = tiles * k_blocks;
    const int64_t g = min64(sm_count, iters);
    auto begin = [&](int64_t c) { return c * iters / g; };
    auto owner = [&](int64_t i) {
        int64_t c = i * g / iters;
        while (c + 1 < g && begin(c + 1) <= i) ++c;
        while (c > 0 && begin(c) > i) --c;
        return c;
    };
    int64_t maxc = 1;
    for (int64_t t = 0; t < tiles; ++t)
        maxc = max64(maxc, owner((t + 1) * k_blocks - 1) - owner(t * k_blocks) + 1);
    sp.stream = true;
    sp.grid = g;
    sp.splits = (int)maxc;
    sp.group = (int)maxc;
    sp.groups = 1;
    sp.kb_per_split = k_blocks;
    sp.tiles = tiles;
    if (maxc > 1) {
        sp.part1_bytes = (size_t)(tiles * maxc * (int64_t)BM * BN * 4);
        sp.counters = (size_t)(tiles + tiles);
    }
    return sp;
}

// K slices per tile.  Units (tile, slice) run one per SM at a time; pick the
// slice count whose units fill the last wave best, discounted by the extra
// traffic of the float32 partial tiles relative to the operand stream.  At
// most SUM_BATCH^2 slices (both reduction levels then take one load batch),
// at least 2 K blocks per slice.
template <int BN>
static SplitPlan split_plan(int64_t tiles, int64_t k_blocks, double stream_bytes, int sm_count,
                            bool force_split, int hint = 0) {
    SplitPlan sp;
    const int64_t smax = min64((int64_t)SUM_BATCH * SUM_BATCH, max64(1, k_blocks / 2));
    double best = -1.0;
    int64_t best_s = 1;
    for (int64_t sl = force_split ? 2 : 1; sl <= max64(smax, force_split ? 2 : 1); ++sl) {
        const int64_t per = ceil_div(k_blocks, sl);
        const int64_t real = ceil_div(k_blocks, per);          // non-empty slices
        const int64_t units = tiles * real;
        const int64_t waves = ceil_div(units, sm_count);
        const double fill = (double)units / (double)(waves * sm_count);
        const double extra = real > 1 ? 2.0 * (double)units * BM * BN * 4 : 0.0;
        const double score = fill * stream_bytes / (stream_bytes + extra);
        if (score > best + 1e-9) {
            best = score;
            best_s = real;
        }
        if (sl >= smax) break;
    }
    if (hint > 0) best_s = min64(hint, min64(k_blocks, (int64_t)SUM_BATCH * SUM_BATCH));
    sp.kb_per_split = ceil_div(k_blocks, best_s);
    sp.splits = (int)ceil_div(k_blocks, sp.kb_per_split);
    int g = 1;
    while ((int64_t)g * g < sp.splits) ++g;
    sp.group = g < SUM_BATCH ? g : SUM_BATCH;
    sp.groups = (int)ceil_div(sp.splits, sp.group);
    sp.tiles = tiles;
    const int64_t tile_bytes = (int64_t)BM * BN * 4;
    if (sp.splits > 1) {
        sp.part1_bytes = (size_t)(tiles * sp.splits * tile_bytes);
        sp.part2_bytes = sp.groups > 1 ? (size_t)(tiles * sp.groups * tile_bytes) : 0;
        sp.counters = (size_t)(tiles * sp.groups + tiles);
    }
    return sp;
}

template <int BN, bool SPLIT, bool SWAP>
static cudaError_t launch_tc(olc_dtype dt, const Problem& pr, int sm_count, cudaStream_t s,
                             const SplitPlan* sp, const Workspace* ws) {
    using C = Cfg<BN>;
    const int64_t a_ld = pr.a_ld ? pr.a_ld : pr.K, b_ld = pr.b_ld ? pr.b_ld : pr.N;
    if (!(SPLIT || SWAP) && BN == 256) {
        // the general tiles read A and B through row pitches (16-byte rows)
        // and store Y at any alignment
        if (!tc_operands_ok(dt, pr, a_ld, b_ld)) return cudaErrorInvalidValue;
    } else if (!tc_shape_ok(dt, pr.N, pr.K) || pr.M >= (1LL << 31) || pr.a_ld || pr.b_ld ||
               pr.y_unaligned) {
        return cudaErrorInvalidValue;
    }
    if (SWAP && pr.M > BN) return cudaErrorInvalidValue;
    // the operands' batch extents: every item offset is a multiple of the
    // matrix size (dense operands), so offset / size is the TMA batch index
    int64_t a_items = 1, b_items = 1;
    for (int d = 0; d < pr.map.rank; ++d) {
        if (pr.map.a_stride[d])
            a_items = max64(a_items, pr.map.a_stride[d] / (pr.M * pr.K) * pr.map.dims[d]);
        if (pr.map.b_stride[d])
            b_items = max64(b_items, pr.map.b_stride[d] / (pr.K * pr.N) * pr.map.dims[d]);
    }
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    const int bf = dt == OLC_BFLOAT16;
    // A with fewer rows than one tile: load only its rows (rounded up to a
    // whole 8-row swizzle group); the MMA's remaining rows of the stage hold
    // stale data and feed only output rows that are never stored
    const uint32_t a_box_rows = (!SWAP && pr.M < BM) ? (uint32_t)ceil_div(pr.M, 8) * 8 : BM;
    if (!SWAP) {
        if (pr.a_trans) {
            if (!encode_3d(&ma, pr.A, bf, pr.M, pr.K, a_items, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        } else if (!encode_3d(&ma, pr.A, bf, pr.K, pr.M, a_items, BK, a_box_rows,
                              CU_TENSOR_MAP_SWIZZLE_128B, a_ld)) {
            return cudaErrorInvalidValue;
        }
        if (pr.b_trans) {
            if (BN != 256) return cudaErrorInvalidValue;
            if (!encode_3d(&mb, pr.B, bf, pr.K, pr.N, b_items, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        } else if (!encode_3d(&mb, pr.B, bf, pr.N, pr.K, b_items, C::BLK_COLS, BK, b_swizzle<BN>(),
                              b_ld)) {
            return cudaErrorInvalidValue;
        }
    } else {
        // MMA operand A from the problem's B (64-column MN-major boxes), MMA
        // operand B from the problem's A (BN rows, K-major)
        if (!encode_3d(&ma, pr.B, bf, pr.N, pr.K, b_items, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (!encode_3d(&mb, pr.A, bf, pr.K, pr.M, a_items, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }

    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = pr.items;
    p.tiles_m = SWAP ? ceil_div(pr.N, BM) : ceil_div(pr.M, BM);
    p.tiles_n = SWAP ? 1 : ceil_div(pr.N, BN);
    p.tiles_per_item = p.tiles_m * p.tiles_n;
    p.total_tiles = p.tiles_per_item * pr.items;
    p.k_blocks = ceil_div(pr.K, BK);
    p.a_item_elems = pr.M * pr.K;
    p.b_item_elems = pr.K * pr.N;
    p.map = pr.map;
    p.Y = pr.Y;
    p.err = device_error_word();
    p.is_bf16 = bf;
    p.splits = 1;
    p.group = 1;
    p.groups = 1;
    p.kb_per_split = p.k_blocks;
    p.stage_tx_bytes = SWAP ? (uint32_t)(A_STAGE_BYTES + BN * BK * 2)
                            : (uint32_t)((pr.a_trans ? BM : a_box_rows) * BK * 2 + C::B_STAGE_BYTES);
    p.a_mn = pr.a_trans;
    p.b_k = pr.b_trans;
    p.y_unaligned = pr.y_unaligned;
    p.epi = pr.epi;
    if ((pr.a_trans || pr.b_trans) && (SWAP || SPLIT)) return cudaErrorInvalidValue;
    if (SPLIT) {
        if (!sp || !ws || !ws->partials || !ws->counters || (sp->splits < 2 && !sp->stream))
            return cudaErrorInvalidValue;
        p.splits = sp->splits;
        p.group = sp->group;
        p.groups = sp->groups;
        p.kb_per_split = sp->kb_per_split;
        p.part1 = static_cast<float*>(ws->partials);
        p.part2 = sp->groups > 1
                      ? reinterpret_cast<float*>(static_cast<char*>(ws->partials) + sp->part1_bytes)
                      : nullptr;
        p.cnt1 = ws->counters;
        p.cnt2 = ws->counters + sp->tiles * sp->groups;
        p.stream = sp->stream ? 1 : 0;
        p.iterations = p.total_tiles * p.k_blocks;
    }
    if (p.total_tiles <= 0) return cudaSuccess;

    const cudaError_t attr_err =
        set_smem_limit(reinterpret_cast<const void*>(tc_gemm_kernel<BN, SPLIT, SWAP>), C::SMEM_BYTES);
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t units = p.total_tiles * p.splits;
    const int64_t grid = p.stream ? sp->grid : min64(units, (int64_t)sm_count);
    return launch_pdl(tc_gemm_kernel<BN, SPLIT, SWAP>, dim3((unsigned)grid), dim3(THREADS),
                      (size_t)C::SMEM_BYTES, s, ma, mb, p);
}

static cudaError_t launch_pair(olc_dtype dt, const Problem& pr, int sm_count, cudaStream_t s) {
    const int64_t a_ld = pr.a_ld ? pr.a_ld : pr.K, b_ld = pr.b_ld ? pr.b_ld : pr.N;
    if (!tc_operands_ok(dt, pr, a_ld, b_ld)) return cudaErrorInvalidValue;
    int64_t a_items = 1, b_items = 1;
    for (int d = 0; d < pr.map.rank; ++d) {
        if (pr.map.a_stride[d])
            a_items = max64(a_items, pr.map.a_stride[d] / (pr.M * pr.K) * pr.map.dims[d]);
        if (pr.map.b_stride[d])
            b_items = max64(b_items, pr.map.b_stride[d] / (pr.K * pr.N) * pr.map.dims[d]);
    }
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    const int bf = dt == OLC_BFLOAT16;
    const bool at = pr.a_trans != 0, bt = pr.b_trans != 0;
    if (!(at ? encode_3d(&ma, pr.A, bf, pr.M, pr.K, a_items, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B)
             : encode_3d(&ma, pr.A, bf, pr.K, pr.M, a_items, BK, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                         a_ld)))
        return cudaErrorInvalidValue;
    // MN-major B with whole 64-column blocks: one 4-D load per K block
    // instead of two 3-D ones (the producer lane issues every load)
    const bool b_blocks = !bt && pr.N % 64 == 0 && encode_b_blocks(&mb, pr.B, bf, pr.N, pr.K, b_items, b_ld);
    if (!b_blocks &&
        !(bt ? encode_3d(&mb, pr.B, bf, pr.K, pr.N, b_items, BK, 128, CU_TENSOR_MAP_SWIZZLE_128B)
             : encode_3d(&mb, pr.B, bf, pr.N, pr.K, b_items, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B,
                         b_ld)))
        return cudaErrorInvalidValue;
    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = pr.items;
    p.k_blocks = ceil_div(pr.K, BK);
    p.a_item_elems = pr.M * pr.K;
    p.b_item_elems = pr.K * pr.N;
    p.map = pr.map;
    p.b_blocks = b_blocks ? 1 : 0;
    p.Y = pr.Y;
    p.err = device_error_word();
    p.is_bf16 = bf;
    p.a_mn = at;
    p.b_k = bt;
    p.y_unaligned = pr.y_unaligned;
    p.epi = pr.epi;
    const int64_t pairs = ceil_div(pr.M, 256) * ceil_div(pr.N, 256) * pr.items;
    if (pairs <= 0) return cudaSuccess;
    const cudaError_t attr_err =
        set_smem_limit(reinterpret_cast<const void*>(pair::tc_pair_kernel<false>), pair::smem_bytes<false>());
    if (attr_err != cudaSuccess) return attr_err;
    // a last partial wave of r tiles on at most half the clusters runs as 2r
    // half tiles (256 x 128): the same work on twice the SMs, so the wave
    // takes about half as long (the 4096 x 4096 projection: 1024 tiles, 13
    // whole waves of 76 and 36 tiles left -> 72 halves)
    const int64_t per_wave = sm_count / 2;
    const int64_t tail = per_wave > 0 ? pairs % per_wave : 0;
    if (!bt && tail > 0 && 2 * tail <= per_wave) p.pair_half_tiles = tail;
    const int64_t units = pairs + p.pair_half_tiles;
    const int64_t clusters = min64(units, per_wave);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(pair::PAIR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::smem_bytes<false>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, pair::tc_pair_kernel<false>, ma, mb, p);
}

// rank-3 map over [1][rows][cols] bytes (cols innermost), box {box_cols,
// box_rows, 1}, 128-byte swizzle
static bool encode_u8(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, 1};
    cuuint64_t strides[2] = {cols, cols * rows};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit float operands on CTA pairs: A [M, K] and the transposed B [N, K]
// (both bytes, K-major), float32 Y; one item
static cudaError_t launch_pair_f8_impl(olc_dtype dt, const Problem& pr, const void* bt, int sm_count,
                                       cudaStream_t s) {
    if (pr.items != 1 || pr.K % 16 != 0 || pr.N % 4 != 0 || pr.M >= (1LL << 31) ||
        pr.N >= (1LL << 31) || pr.K >= (1LL << 31))
        return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    if (!encode_u8(&ma, pr.A, (uint64_t)pr.K, (uint64_t)pr.M, 128, 128) ||
        !encode_u8(&mb, bt, (uint64_t)pr.K, (uint64_t)pr.N, 128, 128))
        return cudaErrorInvalidValue;
    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = 1;
    p.k_blocks = ceil_div(pr.K, 128);
    p.a_item_elems = pr.M * pr.K;
    p.b_item_elems = pr.K * pr.N;
    p.map = pr.map;
    p.Y = pr.Y;
    p.err = device_error_word();
    p.f8_fmt = dt == OLC_FLOAT8E4M3FN ? 0 : 1;
    p.a_mn = 0;
    p.b_k = 1;
    p.epi = pr.epi;
    const int64_t pairs = ceil_div(pr.M, 256) * ceil_div(pr.N, 256);
    if (pairs <= 0) return cudaSuccess;
    const cudaError_t attr_err =
        set_smem_limit(reinterpret_cast<const void*>(pair::tc_pair_kernel<true>), pair::smem_bytes<true>());
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t clusters = min64(pairs, (int64_t)(sm_count / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(pair::PAIR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::smem_bytes<true>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, pair::tc_pair_kernel<true>, ma, mb, p);
}

// Split-K for tiny outputs: one slice per CTA, clusters of CL CTAs, about one
// CTA per SM (as many clusters as fit at once), slices of at least 2 chunks.
template <int CL>
static cudaError_t tiny_attr() {
    return set_smem_limit(reinterpret_cast<const void*>(tiny::splitk_tiny_kernel<CL>), tiny::SMEM_BYTES);
}

// Clusters of CL that the device runs at once (an estimate from the SM count
// when the occupancy query is unavailable); cached per device.
template <int CL>
static int tiny_max_clusters(int sm_count) {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        dev = -1;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (dev >= 0 && tiny_attr<CL>() == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(CL * (sm_count / CL > 0 ? sm_count / CL : 1)), 1, 1);
        cfg.blockDim = dim3(tiny::THREADS_T, 1, 1);
        cfg.dynamicSmemBytes = tiny::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, tiny::splitk_tiny_kernel<CL>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    }
    if (n <= 0) return sm_count / CL > 0 ? sm_count / CL : 1;
    if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

static int tiny_cluster_size(int64_t slices) { return slices >= 16 ? 8 : (slices >= 8 ? 4 : 2); }

static SplitPlan tiny_plan(const Problem& pr, int sm_count) {
    SplitPlan sp;
    const int64_t kbs = ceil_div(pr.K, BK);
    int64_t want = max64(1, kbs / 2);
    if (pr.split_hint > 0) want = min64(pr.split_hint, kbs);
    const int cl = tiny_cluster_size(want);
    int64_t clusters = max64(1, want / cl);
    if (pr.split_hint <= 0) {
        const int fit = cl == 8 ? tiny_max_clusters<8>(sm_count)
                                : (cl == 4 ? tiny_max_clusters<4>(sm_count) : tiny_max_clusters<2>(sm_count));
        clusters = max64(1, min64(clusters, fit));
    }
    sp.splits = (int)(clusters * cl);
    sp.kb_per_split = ceil_div(kbs, sp.splits);
    sp.group = cl;
    sp.groups = (int)clusters;
    sp.tiles = 1;
    sp.part1_bytes = (size_t)(clusters * tiny::TILE_BYTES);
    sp.part2_bytes = 0;
    sp.counters = (size_t)cl;
    return sp;
}

template <int CL>
static cudaError_t launch_tiny_cl(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p,
                                  int grid, cudaStream_t s) {
    const cudaError_t e = tiny_attr<CL>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(tiny::THREADS_T, 1, 1);
    cfg.dynamicSmemBytes = tiny::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the prologue may overlap the tail of the previous kernel in the stream;
    // the kernel waits for that kernel before touching global memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tiny::splitk_tiny_kernel<CL>, ma, mb, p);
}

static cudaError_t launch_tiny(olc_dtype dt, const Problem& pr, int sm_count, const Workspace& ws,
                               cudaStream_t s) {
    const SplitPlan sp = tiny_plan(pr, sm_count);
    if (ws.partial_bytes < sp.part1_bytes || ws.counter_count < sp.counters || !ws.partials ||
        !ws.counters)
        return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    const int bf = dt == OLC_BFLOAT16;
    if (!encode_3d(&ma, pr.A, bf, pr.K, pr.M, 1, BK, tiny::ROWS, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_3d(&mb, pr.B, bf, pr.N, pr.K, 1, tiny::COLS, BK, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = 1;
    p.k_blocks = ceil_div(pr.K, BK);
    p.Y = pr.Y;
    p.err = device_error_word();
    p.is_bf16 = bf;
    p.epi = pr.epi;
    p.splits = sp.splits;
    p.group = sp.group;
    p.groups = sp.groups;
    p.kb_per_split = sp.kb_per_split;
    p.part1 = static_cast<float*>(ws.partials);
    p.cnt1 = ws.counters;
    switch (sp.group) {
        case 8: return launch_tiny_cl<8>(ma, mb, p, sp.splits, s);
        case 4: return launch_tiny_cl<4>(ma, mb, p, sp.splits, s);
        default: return launch_tiny_cl<2>(ma, mb, p, sp.splits, s);
    }
}

static double operand_bytes(const Problem& pr) {
    // A and B streamed once per item (upper bound for broadcast operands)
    return 2.0 * (double)(pr.M * pr.K + pr.K * pr.N) * (double)pr.items;
}

// Clusters of `ways` CTAs of the cluster split-K kernel that fit on the GPU
// at once (one CTA per SM; a cluster takes its SMs from one GPC, so fewer
// fit than the SM count suggests); queried once per size and device
static int csplit_max_clusters(int ways, int sm_count) {
    static std::mutex mu;
    static int cached[64][csplit::MAX_WAYS + 1];
    static bool done[64][csplit::MAX_WAYS + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return sm_count / ways / 2;                 // no device: a conservative guess
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev][ways]) {
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ways, 1, 1);
        cfg.blockDim = dim3(csplit::THREADS_CS, 1, 1);
        cfg.dynamicSmemBytes = csplit::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)ways;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (set_smem_limit(reinterpret_cast<const void*>(csplit::csplit_kernel), csplit::SMEM_BYTES) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, csplit::csplit_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = sm_count / ways / 2;
        }
        cached[dev][ways] = n;
        done[dev][ways] = true;
    }
    return cached[dev][ways];
}

// K slices per tile: the most (at most 8, at least 2 K blocks each, no
// slice empty) whose tiles x slices CTAs fit the SMs and whose clusters all
// run in one wave
static int csplit_ways(olc_dtype dt, const Problem& pr, int sm_count) {
    if (!(dt == OLC_FLOAT16 || dt == OLC_BFLOAT16) || pr.a_trans || pr.b_trans || pr.a_ld || pr.b_ld ||
        pr.y_unaligned || !tc_shape_ok(dt, pr.N, pr.K) || pr.M >= (1LL << 31))
        return 0;
    const int64_t tiles = ceil_div(pr.M, BM) * ceil_div(pr.N, csplit::BN) * pr.items;
    const int64_t kbs = ceil_div(pr.K, BK);
    if (tiles <= 0 || 2 * tiles > (int64_t)sm_count) return 0;
    const int64_t wmax = min64(min64((int64_t)sm_count / tiles, (int64_t)csplit::MAX_WAYS), kbs / 2);
    for (int64_t w = wmax; w >= 2; --w) {
        const int64_t ways = ceil_div(kbs, ceil_div(kbs, w));     // no empty slice
        if (ways < 2) break;
        if (tiles > csplit_max_clusters((int)ways, sm_count)) continue;
        // two slices double the streaming CTAs but add the partial tiles'
        // traffic to an already HBM-bound B stream: worth it only for few
        // rows (BF16 [128, 4096] x [4096, 14336]: 31.6 us against 28.1 on
        // CTA pairs; [17, ...]: 23.5 against 26.7)
        if (ways == 2 && pr.M > 64) return 0;
        return (int)ways;
    }
    return 0;
}

static cudaError_t launch_csplit(olc_dtype dt, const Problem& pr, int ways, float* partials, cudaStream_t s) {
    int64_t a_items = 1, b_items = 1;
    for (int d = 0; d < pr.map.rank; ++d) {
        if (pr.map.a_stride[d])
            a_items = max64(a_items, pr.map.a_stride[d] / (pr.M * pr.K) * pr.map.dims[d]);
        if (pr.map.b_stride[d])
            b_items = max64(b_items, pr.map.b_stride[d] / (pr.K * pr.N) * pr.map.dims[d]);
    }
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    const int bf = dt == OLC_BFLOAT16;
    // A with fewer rows than one tile: only its rows are loaded (rounded up
    // to a whole 8-row swizzle group); the stage's other rows feed only
    // output rows that are never stored
    const uint32_t a_box_rows = pr.M < BM ? (uint32_t)ceil_div(pr.M, 8) * 8 : BM;
    if (!encode_3d(&ma, pr.A, bf, pr.K, pr.M, a_items, BK, a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const bool b_blocks = pr.N % 64 == 0 && encode_b_blocks(&mb, pr.B, bf, pr.N, pr.K, b_items, pr.N, 4);
    if (!b_blocks && !encode_3d(&mb, pr.B, bf, pr.N, pr.K, b_items, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = pr.items;
    p.tiles_m = ceil_div(pr.M, BM);
    p.tiles_n = ceil_div(pr.N, csplit::BN);
    p.tiles_per_item = p.tiles_m * p.tiles_n;
    p.total_tiles = p.tiles_per_item * pr.items;
    p.k_blocks = ceil_div(pr.K, BK);
    p.a_item_elems = pr.M * pr.K;
    p.b_item_elems = pr.K * pr.N;
    p.map = pr.map;
    p.b_blocks = b_blocks ? 1 : 0;
    p.Y = pr.Y;
    p.err = device_error_word();
    p.is_bf16 = bf;
    p.stage_tx_bytes = a_box_rows * BK * 2 + csplit::B_BYTES;
    p.epi = pr.epi;
    p.part1 = partials;
    if (p.total_tiles <= 0) return cudaSuccess;
    const int64_t kb_per = ceil_div(p.k_blocks, (int64_t)ways);
    if (ceil_div(p.k_blocks, kb_per) != ways || p.total_tiles * ways > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(csplit::csplit_kernel), csplit::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.total_tiles * ways), 1, 1);
    cfg.blockDim = dim3(csplit::THREADS_CS, 1, 1);
    cfg.dynamicSmemBytes = csplit::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ways;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, csplit::csplit_kernel, ma, mb, p, ways, kb_per);
}

}  // namespace tc

// Row-pitch staging copy for operands the TMA cannot read in place: each
// thread writes one 16-byte group of a destination row, loading its source
// elements with the widest accesses the source address allows (the source
// rows are dense with any 2-byte alignment).
__global__ void pad_rows16_kernel(const unsigned short* __restrict__ src, uint4* __restrict__ dst,
                                  int64_t rows, int64_t cols, int64_t pitch) {
    const int64_t groups_per_row = pitch / 8;
    const int64_t total = rows * groups_per_row;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = g / groups_per_row;
        const int64_t c0 = (g - r * groups_per_row) * 8;
        const unsigned short* s = src + r * cols + c0;
        uint32_t w[4];
        if (c0 + 8 <= cols && (reinterpret_cast<uintptr_t>(s) & 3) == 0) {
            const uint32_t* s4 = reinterpret_cast<const uint32_t*>(s);
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = __ldg(s4 + j);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t lo = c0 + 2 * j < cols ? __ldg(s + 2 * j) : 0u;
                const uint32_t hi = c0 + 2 * j + 1 < cols ? __ldg(s + 2 * j + 1) : 0u;
                w[j] = lo | (hi << 16);
            }
        }
        dst[g] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_pad_rows16(const void* src, void* dst, int64_t rows, int64_t cols, int64_t pitch,
                              cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (pitch % 8 != 0 || pitch < cols || (reinterpret_cast<uintptr_t>(dst) & 15) ||
        (reinterpret_cast<uintptr_t>(src) & 1))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t total = rows * (pitch / 8);
    const int64_t blocks = min64(ceil_div(total, 256), (int64_t)sms * 8);
    pad_rows16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const unsigned short*>(src),
                                                            static_cast<uint4*>(dst), rows, cols, pitch);
    return cudaGetLastError();
}

bool tc_shape_ok(olc_dtype dt, int64_t N, int64_t K) {
    if (dt != OLC_FLOAT16 && dt != OLC_BFLOAT16) return false;
    // TMA needs 16-byte row strides; coordinates fit in int32
    return N % 8 == 0 && K % 8 == 0 && N < (1LL << 31) && K < (1LL << 31);
}

cudaError_t launch_pair_f8(olc_dtype dt, const Problem& pr, const void* bt, int sm_count,
                           cudaStream_t s) {
    return tc::launch_pair_f8_impl(dt, pr, bt, sm_count, s);
}

int tc_general_csplit_ways(olc_dtype dt, const Problem& p, int sm_count) {
    return tc::csplit_ways(dt, p, sm_count);
}

size_t tc_general_partial_bytes(olc_dtype dt, const Problem& p, int sm_count) {
    const int ways = tc::csplit_ways(dt, p, sm_count);
    if (ways < 2) return 0;
    const int64_t tiles = ceil_div(p.M, tc::BM) * ceil_div(p.N, tc::csplit::BN) * p.items;
    return (size_t)(tiles * ways) * tc::BM * tc::csplit::BN * sizeof(float);
}

cudaError_t launch_general_tc(olc_dtype dt, const Problem& pr, int sm_count, cudaStream_t s,
                              int variant, const Workspace* ws) {
    // variant 2: CTA pairs with 256 x 256 tiles; 1: one CTA per 128 x 256
    // tile; 0 (automatic): the cluster split-K when its slices apply and the
    // workspace holds their partial tiles, else pairs when N >= 256
    if (variant == 0) {
        const int ways = pr.tc_ways == 0 ? tc::csplit_ways(dt, pr, sm_count) : (pr.tc_ways >= 2 ? pr.tc_ways : 0);
        const int64_t tiles = ceil_div(pr.M, tc::BM) * ceil_div(pr.N, tc::csplit::BN) * pr.items;
        const size_t need = (size_t)(tiles * (ways > 0 ? ways : 0)) * tc::BM * tc::csplit::BN * sizeof(float);
        if (ways >= 2 && ws && ws->partials && ws->partial_bytes >= need)
            return tc::launch_csplit(dt, pr, ways, static_cast<float*>(ws->partials), s);
    }
    // CTA pairs whenever N holds a pair tile: the spare rows of a 256-row
    // pair tile cost less than leaving half the SMs of a 128-row band idle
    // (BF16 x [4096, 14336], us, pairs / one CTA per 128 x 256 tile: 17
    // rows 26.8 / 30.3, 128 rows 27.9 / 32.9, 255 rows 28.8 / 33.7)
    const bool pair = variant == 2 || (variant == 0 && pr.N >= 256);
    if (pair && sm_count >= 2) return tc::launch_pair(dt, pr, sm_count, s);
    return tc::launch_tc<256, false, false>(dt, pr, sm_count, s, nullptr, nullptr);
}

// skinny-N: 16-column tiles; when the row tiles leave most SMs idle,
// stream-K shares of the K blocks keep every SM streaming A
static tc::SplitPlan tc_skinny_n_plan(const Problem& pr, int sm_count) {
    const int64_t tiles = ceil_div(pr.M, tc::BM) * pr.items;
    const int64_t kbs = ceil_div(pr.K, tc::BK);
    // stream-K only when the row tiles fill at most half the SMs: with more
    // tiles the stream is bound by DRAM, not by idle SMs, and the partials
    // only add traffic
    if (pr.split_hint == 1 || 2 * tiles > (int64_t)sm_count || kbs < 2) {
        tc::SplitPlan none;
        none.tiles = tiles;
        return none;
    }
    tc::SplitPlan sp = tc::stream_plan<16>(tiles, kbs, sm_count);
    if (sp.splits > tc::SUM_BATCH) {
        tc::SplitPlan none;
        none.tiles = tiles;
        return none;
    }
    return sp;
}

size_t tc_skinny_n_partial_bytes(const Problem& pr, int sm_count) {
    return tc_skinny_n_plan(pr, sm_count).part1_bytes;
}

size_t tc_skinny_n_counter_count(const Problem& pr, int sm_count) {
    return tc_skinny_n_plan(pr, sm_count).counters;
}

cudaError_t launch_skinny_n_tc(olc_dtype dt, const Problem& pr, int sm_count, const Workspace& ws,
                               cudaStream_t s) {
    if (pr.N > 16) return cudaErrorInvalidValue;
    const tc::SplitPlan sp = tc_skinny_n_plan(pr, sm_count);
    if (!sp.stream || sp.part1_bytes == 0)
        return tc::launch_tc<16, false, false>(dt, pr, sm_count, s, nullptr, nullptr);
    if (ws.partial_bytes < sp.part1_bytes || ws.counter_count < sp.counters)
        return cudaErrorInvalidValue;
    return tc::launch_tc<16, true, false>(dt, pr, sm_count, s, &sp, &ws);
}

// ---- split-K on the tensor cores: tile width by N
static int tc_split_bn(int64_t N) { return N <= 16 ? 16 : (N <= 32 ? 32 : 256); }

// outputs of at most 32 x 32 (one item): the mma.sync split-K kernel
static bool tc_split_tiny(const Problem& pr) { return pr.M <= 32 && pr.N <= 32 && pr.items == 1; }

static tc::SplitPlan tc_split_plan(const Problem& pr, int sm_count) {
    if (tc_split_tiny(pr)) return tc::tiny_plan(pr, sm_count);
    const int bn = tc_split_bn(pr.N);
    const int64_t tiles = ceil_div(pr.M, tc::BM) * ceil_div(pr.N, bn) * pr.items;
    const int64_t kbs = ceil_div(pr.K, tc::BK);
    const double bytes = tc::operand_bytes(pr);
    switch (bn) {
        case 16: return tc::split_plan<16>(tiles, kbs, bytes, sm_count, true, pr.split_hint);
        case 32: return tc::split_plan<32>(tiles, kbs, bytes, sm_count, true, pr.split_hint);
        default: return tc::split_plan<256>(tiles, kbs, bytes, sm_count, true, pr.split_hint);
    }
}

int tc_split_pick(const Problem& pr, int sm_count) { return tc_split_plan(pr, sm_count).splits; }

size_t tc_split_partial_bytes(const Problem& pr, int sm_count) {
    const tc::SplitPlan sp = tc_split_plan(pr, sm_count);
    return sp.part1_bytes + sp.part2_bytes;
}

size_t tc_split_counter_count(const Problem& pr, int sm_count) {
    return tc_split_plan(pr, sm_count).counters;
}

cudaError_t launch_tc_split(olc_dtype dt, const Problem& pr, int sm_count, const Workspace& ws,
                            cudaStream_t s) {
    if (tc_split_tiny(pr)) return tc::launch_tiny(dt, pr, sm_count, ws, s);
    const tc::SplitPlan sp = tc_split_plan(pr, sm_count);
    if (sp.splits < 2) {
        // a K too short to split: the plain tile kernel of the same width
        switch (tc_split_bn(pr.N)) {
            case 16: return tc::launch_tc<16, false, false>(dt, pr, sm_count, s, nullptr, nullptr);
            case 32: return tc::launch_tc<32, false, false>(dt, pr, sm_count, s, nullptr, nullptr);
            default: return tc::launch_tc<256, false, false>(dt, pr, sm_count, s, nullptr, nullptr);
        }
    }
    if (ws.partial_bytes < sp.part1_bytes + sp.part2_bytes || ws.counter_count < sp.counters)
        return cudaErrorInvalidValue;
    switch (tc_split_bn(pr.N)) {
        case 16: return tc::launch_tc<16, true, false>(dt, pr, sm_count, s, &sp, &ws);
        case 32: return tc::launch_tc<32, true, false>(dt, pr, sm_count, s, &sp, &ws);
        default: return tc::launch_tc<256, true, false>(dt, pr, sm_count, s, &sp, &ws);
    }
}

// ---- skinny-M on the tensor cores: Y^T = B^T A^T, 128 output columns per
// tile along the MMA's M side, the (at most 16) output rows along its N side
static tc::SplitPlan tc_skinny_m_plan(const Problem& pr, int sm_count) {
    const int64_t tiles = ceil_div(pr.N, tc::BM) * pr.items;
    return tc::split_plan<16>(tiles, ceil_div(pr.K, tc::BK), tc::operand_bytes(pr), sm_count,
                              false, pr.split_hint);
}

int tc_skinny_m_pick(const Problem& pr, int sm_count) { return tc_skinny_m_plan(pr, sm_count).splits; }

size_t tc_skinny_m_partial_bytes(const Problem& pr, int sm_count) {
    const tc::SplitPlan sp = tc_skinny_m_plan(pr, sm_count);
    return sp.part1_bytes + sp.part2_bytes;
}

size_t tc_skinny_m_counter_count(const Problem& pr, int sm_count) {
    return tc_skinny_m_plan(pr, sm_count).counters;
}

cudaError_t launch_tc_skinny_m(olc_dtype dt, const Problem& pr, int sm_count, const Workspace& ws,
                               cudaStream_t s) {
    if (pr.M > 16) return cudaErrorInvalidValue;
    const tc::SplitPlan sp = tc_skinny_m_plan(pr, sm_count);
    if (sp.splits < 2) return tc::launch_tc<16, false, true>(dt, pr, sm_count, s, nullptr, nullptr);
    if (ws.partial_bytes < sp.part1_bytes + sp.part2_bytes || ws.counter_count < sp.counters)
        return cudaErrorInvalidValue;
    return tc::launch_tc<16, true, true>(dt, pr, sm_count, s, &sp, &ws);
}

}  // namespace olc

namespace olc {
namespace tc {

// One thread: an mbarrier that expects one arrival, which is made only when
// `arrive` is set; then the same bounded wait the GEMM kernel uses.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int arrive, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive) mbar_arrive(&bar);
    mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace tc
}  // namespace olc

extern "C" olc_status olc_debug_wait_selftest(uint64_t limit_ns, int arrive, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    olc::tc::wait_selftest_kernel<<<1, 1, 0, s>>>((unsigned long long)limit_ns, arrive,
                                                  olc::device_error_word());
    if (cudaGetLastError() != cudaSuccess) return OLC_ERR_CUDA;
    unsigned int flags = 0;
    if (olc::read_and_clear_device_error(&flags, s) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    return flags ? OLC_ERR_DEVICE_TIMEOUT : OLC_OK;
}

extern "C" uint64_t olc_debug_tc_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                           uint32_t layout) {
    return olc::tc::smem_desc(addr, lbo, sbo, layout);
}
extern "C" uint32_t olc_debug_tc_instr_desc(int is_bf16, int m, int n, int a_mn_major,
                                            int b_mn_major) {
    return olc::tc::instr_desc(is_bf16, m, n, a_mn_major, b_mn_major);
}
