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

#include <cstring>
#include <mutex>

#include "common.cuh"

namespace olc {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;               // one 128-byte swizzle span of 16-bit elements
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int A_STAGE_BYTES = BM * BK * 2;       // 16 KiB
constexpr int B_STAGE_BYTES = BN * BK * 2;       // 32 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int ACC_COLS = BN;                     // float32 columns per accumulator
constexpr int TMEM_COLS = 2 * ACC_COLS;          // 512: double buffer
constexpr int THREADS = 192;
constexpr int GROUP_M = 16;                      // tile raster: 16 M-blocks per group
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

struct Smem {
    // stage buffers come first (1024-byte aligned), barriers after
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* alignment slack */ + 256;

struct Params {
    int64_t M, N, K;          // per batch item
    int64_t items;
    int64_t tiles_m, tiles_n, tiles_per_item, total_tiles;
    int64_t k_blocks;
    int64_t a_item_elems;     // M * K: A matrix size (for the TMA batch coordinate)
    int64_t b_item_elems;     // K * N
    BatchMap map;
    void* Y;
    unsigned int* err;
    int is_bf16;
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

// Bounded wait: returns false when the wait ran out or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
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

// ---------------------------------------------------------------------------
// descriptors (host and device agree on these encodings; the host unit test
// checks them bit by bit)

// Shared-memory matrix descriptor for tcgen05: start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// the fixed value 1 in bits 46-47, base offset 0 in 49-51, relative LBO mode
// (bit 52 = 0), swizzle mode in 61-63 (2 = 128-byte swizzle).
__host__ __device__ constexpr uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16: float32 accumulator (bits 4-5 = 1),
// A and B type in bits 7-9 / 10-12 (0 = F16, 1 = BF16), A K-major (bit 15 =
// 0), B MN-major (bit 16 = 1), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(int is_bf16, int m, int n, int b_mn_major) {
    return (1u << 4) | ((uint32_t)is_bf16 << 7) | ((uint32_t)is_bf16 << 10) |
           ((uint32_t)b_mn_major << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
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

__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_b, const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned stage buffers (the 128-byte swizzle pattern repeats
    // every 1024 bytes and the descriptors assume an aligned base)
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem* s = reinterpret_cast<Smem*>(base + STAGES * STAGE_BYTES);
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
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(&s->tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed_parity[STAGES];
            bool armed[STAGES];
            for (int i = 0; i < STAGES; ++i) armed[i] = false;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                int64_t item, mb, nb;
                tile_coords(p, t, item, mb, nb);
                int64_t a_off, b_off;
                batch_offsets(p.map, item, a_off, b_off);
                const int a_item = (int)(a_off / p.a_item_elems);
                const int b_item = (int)(b_off / p.b_item_elems);
                const int m0 = (int)(mb * BM), n0 = (int)(nb * BN);
                for (int64_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&s->empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    unsigned char* sa = base + stage * STAGE_BYTES;
                    unsigned char* sb = sa + A_STAGE_BYTES;
                    mbar_arrive_expect_tx(&s->full[stage], STAGE_BYTES);
                    armed[stage] = true;
                    armed_parity[stage] = phase;
                    const int k0 = (int)(kb * BK);
                    tma_load_3d(sa, &tmap_a, &s->full[stage], k0, m0, a_item);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_3d(sb + j * (64 * BK * 2), &tmap_b, &s->full[stage], n0 + 64 * j,
                                    k0, b_item);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (*abort_flag) {
                // let this CTA's own loads land before the CTA goes away
                for (int i = 0; i < STAGES; ++i)
                    if (armed[i]) mbar_wait_drain(&s->full[i], armed_parity[i]);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc(p.is_bf16, BM, BN, 1);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&s->acc_empty[acc], acc_phase ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                for (int64_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&s->full[stage], phase, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(base + stage * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        // A: K-major, advance 16 elements = 32 bytes inside the swizzle row
                        const uint64_t ad = smem_desc(a_addr + kk * UMMA_K * 2, 16, 1024);
                        // B: MN-major, advance 16 K-rows = 2048 bytes; 64-column
                        // blocks 8192 bytes apart (LBO), 8-row groups 1024 (SBO)
                        const uint64_t bd = smem_desc(b_addr + kk * UMMA_K * 128, 64 * BK * 2, 1024);
                        mma_f16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
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
        uint32_t acc = 0, acc_phase = 0;
        for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
            int64_t item, mb, nb;
            tile_coords(p, t, item, mb, nb);
            if (!mbar_wait(&s->acc_full[acc], acc_phase, abort_flag, p.err)) break;
            tc_fence_after();
            const int64_t row = mb * BM + row_in_tile;
            const bool row_ok = row < p.M;
            const uint32_t t_base = tmem_base + ((uint32_t)(lane_group * 32) << 16) + acc * ACC_COLS;
            unsigned char* yrow = static_cast<unsigned char*>(p.Y) +
                                  ((item * p.M + (row_ok ? row : 0)) * p.N) * 2;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c, r);
                const int64_t col = nb * BN + c;
                if (row_ok && col < p.N) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float lo = __uint_as_float(r[2 * i]);
                        const float hi = __uint_as_float(r[2 * i + 1]);
                        if (p.is_bf16) {
                            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
                            packed[i] = *reinterpret_cast<uint32_t*>(&v);
                        } else {
                            __half2 v = __floats2half2_rn(lo, hi);
                            packed[i] = *reinterpret_cast<uint32_t*>(&v);
                        }
                    }
                    uint4* dst = reinterpret_cast<uint4*>(yrow + col * 2);
                    if (col + 32 <= p.N) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                                packed[4 * q + 3]);
                    } else {
                        // N is a multiple of 8: whole 16-byte groups only
                        const int groups = (int)((p.N - col) / 8);
                        for (int q = 0; q < groups; ++q)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                                packed[4 * q + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s->acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

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
// 128-byte swizzle, box {box_cols, box_rows, 1}
static bool encode_3d(CUtensorMap* map, const void* base, int is_bf16, uint64_t cols,
                      uint64_t rows, uint64_t items, uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, items};
    cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_shape_ok(olc_dtype dt, int64_t N, int64_t K) {
    if (dt != OLC_FLOAT16 && dt != OLC_BFLOAT16) return false;
    // TMA needs 16-byte row strides; coordinates fit in int32
    return N % 8 == 0 && K % 8 == 0 && N < (1LL << 31) && K < (1LL << 31);
}

cudaError_t launch_general_tc(olc_dtype dt, const Problem& pr, int sm_count, cudaStream_t s) {
    using namespace tc;
    if (!tc_shape_ok(dt, pr.N, pr.K) || pr.M >= (1LL << 31)) return cudaErrorInvalidValue;
    // the operands' batch extents: every item offset is a multiple of the
    // matrix size (dense operands), so offset / size is the TMA batch index
    int64_t a_items = 1, b_items = 1;
    for (int d = 0; d < pr.map.rank; ++d) {
        if (pr.map.a_stride[d]) a_items = max64(a_items, pr.map.a_stride[d] / (pr.M * pr.K) * pr.map.dims[d]);
        if (pr.map.b_stride[d]) b_items = max64(b_items, pr.map.b_stride[d] / (pr.K * pr.N) * pr.map.dims[d]);
    }
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    const int bf = dt == OLC_BFLOAT16;
    if (!encode_3d(&ma, pr.A, bf, pr.K, pr.M, a_items, BK, BM)) return cudaErrorInvalidValue;
    if (!encode_3d(&mb, pr.B, bf, pr.N, pr.K, b_items, 64, BK)) return cudaErrorInvalidValue;

    Params p;
    std::memset(&p, 0, sizeof p);
    p.M = pr.M;
    p.N = pr.N;
    p.K = pr.K;
    p.items = pr.items;
    p.tiles_m = ceil_div(pr.M, BM);
    p.tiles_n = ceil_div(pr.N, BN);
    p.tiles_per_item = p.tiles_m * p.tiles_n;
    p.total_tiles = p.tiles_per_item * pr.items;
    p.k_blocks = ceil_div(pr.K, BK);
    p.a_item_elems = pr.M * pr.K;
    p.b_item_elems = pr.K * pr.N;
    p.map = pr.map;
    p.Y = pr.Y;
    p.err = device_error_word();
    p.is_bf16 = bf;
    if (p.total_tiles <= 0) return cudaSuccess;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t grid = min64(p.total_tiles, (int64_t)sm_count);
    tc_gemm_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, s>>>(ma, mb, p);
    return cudaGetLastError();
}

}  // namespace olc

extern "C" uint64_t olc_debug_tc_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return olc::tc::smem_desc(addr, lbo, sbo);
}
extern "C" uint32_t olc_debug_tc_instr_desc(int is_bf16, int m, int n, int b_mn_major) {
    return olc::tc::instr_desc(is_bf16, m, n, b_mn_major);
}
