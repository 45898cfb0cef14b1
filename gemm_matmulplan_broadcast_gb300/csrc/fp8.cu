// MatMul of 8-bit float operands (E4M3FN, E5M2) with float32 accumulation
// and a FLOAT output.
//
// "Gemm and MatMul Performance Roadmap", the Float8 packing-format item: the
// Float8 formats are packing formats whose one-byte patterns decode exactly
// to float32, with float32 accumulation.  On GB300 the tensor cores take the
// two formats directly (tcgen05.mma kind::f8f6f4, float32 accumulator in
// TMEM), so no decode pass exists on the fast path; the SIMT kernel (any
// shape or batch) decodes each byte from its fields.
//
// Fast path: B is first transposed ([K, N] -> [N, K], bytes, through shared
// memory) into the plan's workspace, so that both operands reach the MMA
// K-major with 128-byte swizzle (128 K-elements per swizzle row, 32 per MMA);
// then a persistent warp-specialised kernel (one TMA lane, one MMA lane that
// owns TMEM, four epilogue warps) computes 128 x 256 tiles with two TMEM
// accumulators, and the epilogue writes float32 rows (plus the optional
// fused residual and activation).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"

namespace olc {

namespace tc {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();   // csrc/tc_gemm.cu
}

namespace f8 {

// ---------------------------------------------------------------------------
// decode

// FMT: 0 E4M3FN, 1 E5M2, 2 E4M3FNUZ, 3 E5M2FNUZ
template <int FMT>
__device__ __forceinline__ float decode(uint32_t b) {
    return fp8_decode<FMT>(b);
}

// ---------------------------------------------------------------------------
// SIMT kernel: 64 x 64 tiles of one batch item, 256 threads, 4 x 4 outputs
// per thread, float32 accumulation

template <int FMT>
__global__ void __launch_bounds__(256)
simt_kernel(Problem p, int64_t tiles_m, int64_t tiles_n) {
    constexpr int BMs = 64, BNs = 64, BKs = 16, TMs = 4, TNs = 4, TX = BNs / TNs, TY = BMs / TMs;
    __shared__ float As[BKs][BMs + 1];
    __shared__ float Bs[BKs][BNs];
    const int64_t per_item = tiles_m * tiles_n;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int64_t m0 = (rem / tiles_n) * BMs, n0 = (rem % tiles_n) * BNs;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const unsigned char* __restrict__ A = static_cast<const unsigned char*>(p.A) + a_off;
    const unsigned char* __restrict__ B = static_cast<const unsigned char*>(p.B) + b_off;
    float* __restrict__ Y = static_cast<float*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;
    const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
    float acc[TMs][TNs];
#pragma unroll
    for (int i = 0; i < TMs; ++i)
#pragma unroll
        for (int j = 0; j < TNs; ++j) acc[i][j] = 0.f;
    for (int64_t k0 = 0; k0 < K; k0 += BKs) {
        for (int e = threadIdx.x; e < BMs * BKs; e += 256) {
            const int r = e / BKs, c = e % BKs;
            const int64_t gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K) ? decode<FMT>(A[gm * K + gk]) : 0.f;
        }
        for (int e = threadIdx.x; e < BKs * BNs; e += 256) {
            const int r = e / BNs, c = e % BNs;
            const int64_t gk = k0 + r, gn = n0 + c;
            Bs[r][c] = (gk < K && gn < N) ? decode<FMT>(B[gk * N + gn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BKs; ++kk) {
            float a[TMs], b[TNs];
#pragma unroll
            for (int i = 0; i < TMs; ++i) a[i] = As[kk][ty + i * TY];
#pragma unroll
            for (int j = 0; j < TNs; ++j) b[j] = Bs[kk][tx + j * TX];
#pragma unroll
            for (int i = 0; i < TMs; ++i)
#pragma unroll
                for (int j = 0; j < TNs; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TMs; ++i) {
        const int64_t gm = m0 + ty + i * TY;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TNs; ++j) {
            const int64_t gn = n0 + tx + j * TX;
            if (gn < N) Y[gm * N + gn] = apply_epilogue<float>(p.epi, acc[i][j], gm, gn, Y + gm * N + gn);
        }
    }
}

// ---------------------------------------------------------------------------
// B transpose: [K, N] bytes -> [N, K] bytes, 64 x 64 tiles through shared memory

__global__ void __launch_bounds__(256) transpose_kernel(const unsigned char* __restrict__ B,
                                                        unsigned char* __restrict__ Bt, int64_t K,
                                                        int64_t N, int64_t tiles_n) {
    __shared__ unsigned char t[64][65];
    const int64_t k0 = (blockIdx.x / tiles_n) * 64, n0 = (blockIdx.x % tiles_n) * 64;
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int r = e / 64, c = e % 64;                   // r: k, c: n (coalesced along n)
        if (k0 + r < K && n0 + c < N) t[r][c] = B[(k0 + r) * N + n0 + c];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int r = e / 64, c = e % 64;                   // r: n, c: k (coalesced along k)
        if (n0 + r < N && k0 + c < K) Bt[(n0 + r) * K + k0 + c] = t[c][r];
    }
}

// Vector form for K % 16 == 0 and N % 16 == 0 (16-byte aligned rows): 128 x
// 128 byte tiles, 16-byte loads along n and 16-byte stores along k.  Tile
// row r keeps its 16-byte chunk c at chunk c ^ ((r >> 4) & 7), so the 32
// lanes of a store warp (8 k-chunks x 4 n) read 32 different banks.
constexpr int TT = 128;

__global__ void __launch_bounds__(256) transpose16_kernel(const unsigned char* __restrict__ B,
                                                          unsigned char* __restrict__ Bt, int64_t K,
                                                          int64_t N, int64_t tiles_n) {
    __shared__ __align__(16) unsigned char t[TT * TT];
    const int64_t k0 = (blockIdx.x / tiles_n) * TT, n0 = (blockIdx.x % tiles_n) * TT;
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid + 256 * i;
        const int r = e >> 3, c = e & 7;                  // r: k, c: 16-byte chunk along n
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k0 + r < K && n0 + c * 16 < N)
            v = __ldg(reinterpret_cast<const uint4*>(B + (k0 + r) * N + n0 + c * 16));
        *reinterpret_cast<uint4*>(t + r * TT + ((c ^ ((r >> 4) & 7)) << 4)) = v;
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    const int kc = lane & 7;                              // 16-byte chunk along k
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = warp * 16 + i * 4 + (lane >> 3);    // tile column = output row
        const int col = ((n >> 4) ^ kc) << 4 | (n & 15);  // rows kc*16.. share (r >> 4) = kc
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = kc * 16 + q * 4;
            w[q] = (uint32_t)t[r * TT + col] | ((uint32_t)t[(r + 1) * TT + col] << 8) |
                   ((uint32_t)t[(r + 2) * TT + col] << 16) | ((uint32_t)t[(r + 3) * TT + col] << 24);
        }
        if (n0 + n < N && k0 + kc * 16 < K)
            *reinterpret_cast<uint4*>(Bt + (n0 + n) * K + k0 + kc * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------------------
// tensor-core kernel

constexpr int BM = 128, BN = 256;
constexpr int BKB = 128;                      // K elements (bytes) per stage: one swizzle row
constexpr int UMMA_K = 32;                    // K per kind::f8f6f4 MMA
constexpr int A_BYTES = BM * BKB;             // 16 KiB
constexpr int B_BYTES = BN * BKB;             // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;             // two float32 accumulators
constexpr int GROUP_M = 16;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr unsigned long long kWaitNs = 4000000000ull;

struct Shared {
    uint64_t full[STAGES], empty[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct Params {
    int64_t M, N, K;
    int64_t tiles_m, tiles_n, total_tiles, k_blocks;
    float* Y;
    unsigned int* err;
    int fmt;                  // 0: E4M3, 1: E5M2 (the kind::f8f6f4 format codes)
    Epilogue epi;
};

__device__ __forceinline__ uint32_t su32(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_expect(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait: false when it ran out (error word set, abort raised) or
// another role aborted
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err) {
    if (bar_try(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (bar_try(b, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            raise_device_error(err, kErrWaitTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ void bar_drain(uint64_t* b, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!bar_try(b, parity))
        if (globaltimer_ns() - t0 > kWaitNs) return;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* b, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(b)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// K-major operand rows of 128 bytes, 128-byte swizzle: start >> 4, LBO 16
// (unused with swizzling), SBO 1024 (8-row groups), version 1 at bit 46,
// layout code 2 at bits 61-63
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(16 >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f8f6f4 instruction descriptor: float32 accumulator (bits 4-5 = 1), A
// and B formats in bits 7-9 / 10-12 (0 = E4M3, 1 = E5M2), both K-major (bits
// 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28
__host__ __device__ constexpr uint32_t f8_instr_desc(int fmt, int m, int n) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tile_of(const Params& p, int64_t t, int64_t& mb, int64_t& nb) {
    const int64_t span = (int64_t)GROUP_M * p.tiles_n;
    const int64_t g = t / span, first = g * GROUP_M;
    const int64_t gm = min64(p.tiles_m - first, GROUP_M);
    const int64_t in = t % span;
    mb = first + in % gm;
    nb = in / gm;
}

__global__ void __launch_bounds__(THREADS, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
          const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared* s = reinterpret_cast<Shared*>(base + STAGES * STAGE_BYTES);
    volatile int* abort_flag = &s->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            bar_init(&s->full[i], 1);
            bar_init(&s->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(&s->acc_full[i], 1);
            bar_init(&s->acc_empty[i], 4);   // one arrival per epilogue warp
        }
        bar_init(&s->drain, 1);
        s->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&s->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = s->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            uint32_t stage = 0, phase = 0;
            bool armed[STAGES];
            uint32_t armed_parity[STAGES];
            for (int i = 0; i < STAGES; ++i) armed[i] = false;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                int64_t mb, nb;
                tile_of(p, t, mb, nb);
                for (int64_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!bar_wait(&s->empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    unsigned char* sa = base + stage * STAGE_BYTES;
                    bar_expect(&s->full[stage], STAGE_BYTES);
                    armed[stage] = true;
                    armed_parity[stage] = phase;
                    const int k0 = (int)(kb * BKB);
                    tma_2d(sa, &tmap_a, &s->full[stage], k0, (int)(mb * BM));
                    tma_2d(sa + A_BYTES, &tmap_b, &s->full[stage], k0, (int)(nb * BN));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (*abort_flag)
                for (int i = 0; i < STAGES; ++i)
                    if (armed[i]) bar_drain(&s->full[i], armed_parity[i]);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = f8_instr_desc(p.fmt, BM, BN);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                if (!bar_wait(&s->acc_empty[acc], acc_phase ^ 1, abort_flag, p.err)) break;
                fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int64_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!bar_wait(&s->full[stage], phase, abort_flag, p.err)) { ok = false; break; }
                    fence_after();
                    const uint32_t a_addr = su32(base + stage * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BKB / UMMA_K; ++kk)
                        mma_f8(d, kmajor_desc(a_addr + kk * UMMA_K), kmajor_desc(b_addr + kk * UMMA_K),
                               idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    commit(&s->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                commit(&s->acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            commit(&s->drain);
            bar_drain(&s->drain, 0);
        }
    } else {
        const int lane_group = warp & 3;
        const int row_in_tile = lane_group * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
            int64_t mb, nb;
            tile_of(p, t, mb, nb);
            if (!bar_wait(&s->acc_full[acc], acc_phase, abort_flag, p.err)) break;
            fence_after();
            const int64_t row = mb * BM + row_in_tile;
            const bool row_ok = row < p.M;
            const uint32_t t_base = tmem_base + ((uint32_t)(lane_group * 32) << 16) + acc * BN;
            float* yrow = p.Y + (row_ok ? row : 0) * p.N;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld32(t_base + c, r);
                const int64_t col = nb * BN + c;
                if (row_ok && col < p.N) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    if (p.epi.mode != 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col + i < p.N)
                                v[i] = apply_epilogue<float>(p.epi, v[i], row, col + i, yrow + col + i);
                    }
                    // N is a multiple of 4: whole 16-byte groups only
                    const int64_t left = (p.N - col) / 4;
                    const int groups = (int)(left < 8 ? left : 8);
                    float4* dst = reinterpret_cast<float4*>(yrow + col);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q < groups) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&s->acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
}

bool encode_u8_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                  uint32_t box_rows) {
    auto fn = tc::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Few rows (M <= 16), E4M3FN / E5M2, B read in its stored layout: the
// tensor cores with swapped operands, Y^T = B^T A^T.  One unit is 128 output
// columns over one K slice; the MMA is kind::f8f6f4 with M = 128 (columns
// n), N = 16 (rows of A, zero-padded), K = 32, float32 accumulators in TMEM.
// The MMA wants both operands K-major, while B is stored [K, N] (n
// contiguous), so B is transposed inside shared memory on the way:
//   warp 0    one lane streams 128 x 128-byte boxes of B (128 K-rows of 128
//             columns, 128-byte swizzle) and 16 x 128-byte boxes of A into
//             an 8-deep ring (full[], empty[]);
//   warps 2-5 transpose each B box into a 2-deep ring of K-major tiles (128
//             rows n of 128 K-bytes, the 128-byte-swizzle layout TMA would
//             write): per 16 x 16-byte block one ldmatrix.x2.trans of byte
//             pairs (its two 8 x 8 matrices take the K rows 4j, 4j + 1 and
//             4j + 2, 4j + 3, so each lane holds two K pairs of two columns),
//             two byte permutes that make four consecutive K bytes of one
//             column, and one stmatrix.x2 (even and odd columns); then they
//             run the epilogue of each unit;
//   warp 1    one lane issues the MMAs (4 per 128-deep block) and owns TMEM
//             (two 16-column accumulators, so a unit's epilogue overlaps the
//             next unit's MMAs).
// K slices: the last slice of a tile to finish sums the tiles' slices in
// slice order (float32 partials in the workspace), so results are the same
// run to run.

namespace sk {

constexpr int TN = 128;                       // output columns per unit (MMA M)
constexpr int KB = 128;                       // K bytes per stage: one swizzle row
constexpr int MR = 16;                        // A rows per MMA (MMA N)
constexpr int RAW_BYTES = KB * TN;            // 16 KiB: B as stored, K rows of 128 columns
constexpr int A_BYTES = MR * KB;              // 2 KiB: A, K-major
constexpr int BT_BYTES = TN * KB;             // 16 KiB: B^T, K-major
constexpr int RING = 8;                       // B / A stages in flight
constexpr int BT_RING = 2;                    // transposed tiles
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 32;                 // two 16-column accumulators
constexpr int SMEM_BYTES = RING * (RAW_BYTES + A_BYTES) + BT_RING * BT_BYTES + 1024 + 512;

struct Bars {
    uint64_t full[RING], empty[RING];
    uint64_t bt_full[BT_RING], bt_empty[BT_RING];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct SkParams {
    int64_t M, N, K;
    int64_t tiles_n, units, kslice;           // kslice: a multiple of KB
    int ksplit;
    float* Y;
    float* part;                              // [tiles_n][ksplit][MR][TN] float32 (ksplit > 1)
    unsigned int* cnt;                        // [tiles_n][4] arrivals per 32-column group, zero between launches
    unsigned int* err;
    int fmt;
    int pre_t;                                // B given transposed ([N, K] bytes): no transposition
    Epilogue epi;
};

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}
__device__ __forceinline__ void stsm_x2(uint32_t addr, uint32_t r0, uint32_t r1) {
    asm volatile("stmatrix.sync.aligned.m8n8.x2.shared.b16 [%0], {%1, %2};" ::"r"(addr), "r"(r0), "r"(r1)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// unit u -> column tile and K slice (consecutive units: consecutive tiles)
__device__ __forceinline__ void unit_of(const SkParams& p, int64_t u, int64_t& tile, int& slice,
                                        int64_t& kb0, int64_t& kb1) {
    tile = u % p.tiles_n;
    slice = (int)(u / p.tiles_n);
    const int64_t k0 = (int64_t)slice * p.kslice;
    const int64_t k1 = min64(p.K, k0 + p.kslice);
    kb0 = k0 / KB;
    kb1 = ceil_div(k1, (int64_t)KB);
}

__global__ void __launch_bounds__(THREADS, 1)
skinny_tc_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_a,
                 const SkParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* raw = base;                                    // RING x RAW_BYTES
    unsigned char* bt = base + RING * RAW_BYTES;                  // BT_RING x BT_BYTES
    unsigned char* as = bt + BT_RING * BT_BYTES;                  // RING x A_BYTES
    Bars* s = reinterpret_cast<Bars*>(as + RING * A_BYTES);
    volatile int* abort_flag = &s->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RING; ++i) {
            bar_init(&s->full[i], 1);
            // four transposer warps and the MMA's commit (the MMA's alone when
            // B comes transposed)
            bar_init(&s->empty[i], p.pre_t ? 1 : 5);
        }
        for (int i = 0; i < BT_RING; ++i) {
            bar_init(&s->bt_full[i], 4);
            bar_init(&s->bt_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(&s->acc_full[i], 1);
            bar_init(&s->acc_empty[i], 4);
        }
        bar_init(&s->drain, 1);
        s->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&s->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = s->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            uint32_t st = 0, ph = 0;
            bool armed[RING];
            uint32_t armed_parity[RING];
            for (int i = 0; i < RING; ++i) armed[i] = false;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int64_t tile, kb0, kb1;
                int slice;
                unit_of(p, u, tile, slice, kb0, kb1);
                for (int64_t kb = kb0; kb < kb1; ++kb) {
                    if (!bar_wait(&s->empty[st], ph ^ 1, abort_flag, p.err)) { ok = false; break; }
                    bar_expect(&s->full[st], RAW_BYTES + A_BYTES);
                    armed[st] = true;
                    armed_parity[st] = ph;
                    if (p.pre_t)   // B^T: 128 rows n of 128 K-bytes, the MMA's layout already
                        tma_2d(raw + st * RAW_BYTES, &tmap_b, &s->full[st], (int)(kb * KB), (int)(tile * TN));
                    else
                        tma_2d(raw + st * RAW_BYTES, &tmap_b, &s->full[st], (int)(tile * TN), (int)(kb * KB));
                    tma_2d(as + st * A_BYTES, &tmap_a, &s->full[st], (int)(kb * KB), 0);
                    if (++st == RING) { st = 0; ph ^= 1; }
                }
            }
            if (*abort_flag)
                for (int i = 0; i < RING; ++i)
                    if (armed[i]) bar_drain(&s->full[i], armed_parity[i]);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = f8_instr_desc(p.fmt, TN, MR);
            uint32_t st = 0, ph = 0, tb = 0, tph = 0, acc = 0, acc_ph = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int64_t tile, kb0, kb1;
                int slice;
                unit_of(p, u, tile, slice, kb0, kb1);
                if (!bar_wait(&s->acc_empty[acc], acc_ph ^ 1, abort_flag, p.err)) break;
                fence_after();
                const uint32_t d = tmem_base + acc * MR;
                for (int64_t kb = kb0; kb < kb1; ++kb) {
                    if ((!p.pre_t && !bar_wait(&s->bt_full[tb], tph, abort_flag, p.err)) ||
                        !bar_wait(&s->full[st], ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    // MMA A: B^T, 128 x 128 K-bytes (transposed here, or as loaded)
                    const uint32_t a_addr = p.pre_t ? su32(raw + st * RAW_BYTES) : su32(bt + tb * BT_BYTES);
                    const uint32_t b_addr = su32(as + st * A_BYTES);      // MMA B: A, 16 x 128 K-bytes
#pragma unroll
                    for (int kk = 0; kk < KB / UMMA_K; ++kk)
                        mma_f8(d, kmajor_desc(a_addr + kk * UMMA_K), kmajor_desc(b_addr + kk * UMMA_K), idesc,
                               (kb > kb0 || kk > 0) ? 1u : 0u);
                    if (!p.pre_t) commit(&s->bt_empty[tb]);
                    commit(&s->empty[st]);
                    if (++st == RING) { st = 0; ph ^= 1; }
                    if (++tb == BT_RING) { tb = 0; tph ^= 1; }
                }
                if (!ok) break;
                commit(&s->acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_ph ^= 1; }
            }
            commit(&s->drain);
            bar_drain(&s->drain, 0);
        }
    } else {
        // ---------------------------------------------------- transpose + epilogue
        const int tw = warp - 2;                  // 0..3
        const int lane_group = warp & 3;          // the TMEM lanes this warp may read
        uint32_t st = 0, ph = 0, tb = 0, tph = 0, acc = 0, acc_ph = 0;
        bool ok = true;
        // this lane's ldmatrix row: matrix (lane >> 3) & 1, row lane & 7 -> K row
        // 4 (row >> 1) + (row & 1) + 2 matrix of a 16-row block
        const int lrow = lane & 7, lmat = (lane >> 3) & 1;
        const int k_in = 4 * (lrow >> 1) + (lrow & 1) + 2 * lmat;    // 0..15
        // stmatrix row: matrix (lane >> 3) & 1 (even / odd column), row lane & 7
        const int n_in = 2 * lrow + lmat;                            // 0..15
        for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int64_t tile, kb0, kb1;
            int slice;
            unit_of(p, u, tile, slice, kb0, kb1);
            for (int64_t kb = kb0; kb < kb1 && !p.pre_t; ++kb) {
                if (!bar_wait(&s->full[st], ph, abort_flag, p.err) ||
                    !bar_wait(&s->bt_empty[tb], tph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t src = su32(raw + st * RAW_BYTES);
                const uint32_t dst = su32(bt + tb * BT_BYTES);
                // 64 blocks of 16 K-rows x 16 columns, 16 per warp
#pragma unroll 4
                for (int b = tw; b < 64; b += 4) {
                    const int kb16 = b >> 3, nb16 = b & 7;
                    // source: K row k, 16-byte chunk nb16 at position nb16 ^ (k & 7)
                    const int k = 16 * kb16 + k_in;
                    uint32_t r0, r1;
                    ldsm_x2_t(src + k * 128 + ((nb16 ^ (k & 7)) << 4), r0, r1);
                    // r0: K rows ka, ka + 1 of columns 2q, 2q + 1; r1: ka + 2, ka + 3
                    // (ka = 4 (lane & 3), q = lane >> 2): four K bytes per column
                    const uint32_t even = __byte_perm(r0, r1, 0x6420);
                    const uint32_t odd = __byte_perm(r0, r1, 0x7531);
                    // destination: row n, 16-byte chunk kb16 at position kb16 ^ (n & 7)
                    const int n = 16 * nb16 + n_in;
                    stsm_x2(dst + n * 128 + ((kb16 ^ (n & 7)) << 4), even, odd);
                }
                // generic-proxy writes, read next by the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    bar_arrive(&s->bt_full[tb]);
                    bar_arrive(&s->empty[st]);
                }
                if (++st == RING) { st = 0; ph ^= 1; }
                if (++tb == BT_RING) { tb = 0; tph ^= 1; }
            }
            if (!ok) break;
            // epilogue of the unit: TMEM lane = output column, column = row of A
            if (!bar_wait(&s->acc_full[acc], acc_ph, abort_flag, p.err)) break;
            fence_after();
            uint32_t r[16];
            tmem_ld16(tmem_base + ((uint32_t)(lane_group * 32) << 16) + acc * MR, r);
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&s->acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_ph ^= 1; }
            const int64_t n = tile * TN + lane_group * 32 + lane;
            const int rows = (int)min64(p.M, MR);
            if (p.ksplit == 1) {
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < MR; ++m)
                        if (m < rows)
                            p.Y[m * p.N + n] =
                                apply_epilogue<float>(p.epi, __uint_as_float(r[m]), m, n, p.Y + m * p.N + n);
                }
                continue;
            }
            // K slices: each warp files its 32 columns of this slice's partial
            // tile and arrives on the counter of its column group; the last of
            // the group's ksplit arrivals sums the slices in slice order.
            // Warps coordinate only through the counters, so no warp can be
            // left waiting for another that gave up.
            const int64_t col = lane_group * 32 + lane;
            float* mine = p.part + ((tile * p.ksplit + slice) * MR) * (int64_t)TN + col;
#pragma unroll
            for (int m = 0; m < MR; ++m)
                if (m < rows) mine[m * TN] = __uint_as_float(r[m]);
            __threadfence();
            __syncwarp();
            unsigned int* c = p.cnt + tile * 4 + lane_group;
            unsigned int last = 0;
            if (lane == 0) last = atomicAdd(c, 1u) == (unsigned int)p.ksplit - 1u ? 1u : 0u;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!last) continue;
            __threadfence();
            const float* first = p.part + (tile * p.ksplit * MR) * (int64_t)TN + col;
            float v[MR];
#pragma unroll
            for (int m = 0; m < MR; ++m) v[m] = 0.f;
            for (int sl = 0; sl < p.ksplit; ++sl) {
                // one slice's rows loaded together: one L2 round trip per slice
                float t[MR];
#pragma unroll
                for (int m = 0; m < MR; ++m)
                    t[m] = m < rows ? __ldcg(first + ((int64_t)sl * MR + m) * TN) : 0.f;
#pragma unroll
                for (int m = 0; m < MR; ++m) v[m] += t[m];
            }
            if (n < p.N) {
#pragma unroll
                for (int m = 0; m < MR; ++m)
                    if (m < rows) p.Y[m * p.N + n] = apply_epilogue<float>(p.epi, v[m], m, n, p.Y + m * p.N + n);
            }
            if (lane == 0) *c = 0u;   // ready for the next launch
        }
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
}

}  // namespace sk

}  // namespace f8

// E4M3FN / E5M2 few-row products the swapped tensor-core kernel takes: one
// item, N and K multiples of 16, 16-byte aligned A and B
bool f8_skinny_tc_ok(olc_dtype dt, const Problem& p) {
    return (dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2) && p.items == 1 && p.M >= 1 && p.M <= 16 &&
           p.N % 16 == 0 && p.K % 16 == 0 && p.N < (1LL << 31) && p.K < (1LL << 31);
}

// K slices: whole waves of one unit per SM, discounted by the partial
// traffic (the same rule as the other skinny kernels)
int f8_skinny_tc_pick(const Problem& p, int sm_count) {
    if (p.split_hint > 0) return (int)min64(p.split_hint, max64(1, p.K / f8::sk::KB));
    const int64_t tiles = ceil_div(p.N, (int64_t)f8::sk::TN);
    const double stream = (double)p.K * (double)p.N;
    const int64_t smax = min64(32, max64(1, p.K / 1024));
    int best = 1;
    double best_score = -1.0;
    for (int64_t sp = 1; sp <= smax; ++sp) {
        const int64_t units = tiles * sp;
        const int64_t waves = ceil_div(units, (int64_t)sm_count);
        const double fill = (double)units / (double)(waves * sm_count);
        const double extra = sp > 1 ? 2.0 * (double)sp * 16.0 * (double)p.N * 4.0 : 0.0;
        const double score = fill * stream / (stream + extra);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = (int)sp;
        }
    }
    return best;
}

size_t f8_skinny_tc_partial_bytes(const Problem& p, int ksplit) {
    if (ksplit <= 1) return 0;
    return (size_t)(ceil_div(p.N, (int64_t)f8::sk::TN) * ksplit * f8::sk::MR * f8::sk::TN * 4);
}

size_t f8_skinny_tc_counter_count(const Problem& p, int ksplit) {
    return ksplit > 1 ? (size_t)ceil_div(p.N, (int64_t)f8::sk::TN) * 4 : 0;
}

cudaError_t launch_f8_skinny_tc(olc_dtype dt, const Problem& p, int ksplit, int sm_count, const Workspace& ws,
                                cudaStream_t s, const void* bt_ready) {
    using namespace f8::sk;
    const void* bsrc = bt_ready ? bt_ready : p.B;
    if (!f8_skinny_tc_ok(dt, p) || (reinterpret_cast<uintptr_t>(p.A) & 15) || (reinterpret_cast<uintptr_t>(bsrc) & 15))
        return cudaErrorInvalidValue;
    if (ksplit < 1) ksplit = 1;
    const int64_t kslice = ceil_div(ceil_div(p.K, (int64_t)ksplit), (int64_t)KB) * KB;
    ksplit = (int)ceil_div(p.K, kslice);                   // non-empty slices
    SkParams q;
    std::memset(&q, 0, sizeof q);
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.tiles_n = ceil_div(p.N, (int64_t)TN);
    q.ksplit = ksplit;
    q.kslice = kslice;
    q.units = q.tiles_n * ksplit;
    q.Y = static_cast<float*>(p.Y);
    q.err = device_error_word();
    q.fmt = dt == OLC_FLOAT8E4M3FN ? 0 : 1;
    q.pre_t = bt_ready ? 1 : 0;
    q.epi = p.epi;
    if (ksplit > 1) {
        if (!ws.partials || ws.partial_bytes < f8_skinny_tc_partial_bytes(p, ksplit) || !ws.counters ||
            ws.counter_count < (size_t)q.tiles_n * 4)
            return cudaErrorInvalidValue;
        q.part = static_cast<float*>(ws.partials);
        q.cnt = ws.counters;
    }
    CUtensorMap mb, ma;
    std::memset(&mb, 0, sizeof mb);
    std::memset(&ma, 0, sizeof ma);
    // B as stored: [K rows][N bytes], boxes of 128 columns x 128 K-rows (or
    // B^T: [N rows][K bytes], boxes of 128 K-bytes x 128 rows); A: [M rows]
    // [K bytes], boxes of 128 K-bytes x 16 rows (rows past M read 0)
    const bool mb_ok = bt_ready ? f8::encode_u8_2d(&mb, bsrc, (uint64_t)p.K, (uint64_t)p.N, KB, TN)
                                : f8::encode_u8_2d(&mb, bsrc, (uint64_t)p.N, (uint64_t)p.K, TN, KB);
    if (!mb_ok || !f8::encode_u8_2d(&ma, p.A, (uint64_t)p.K, (uint64_t)p.M, KB, MR)) return cudaErrorInvalidValue;
    const cudaError_t attr = set_smem_limit(reinterpret_cast<const void*>(skinny_tc_kernel), SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const int64_t grid = min64(q.units, (int64_t)sm_count);
    skinny_tc_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, s>>>(mb, ma, q);
    return cudaGetLastError();
}

bool fp8_tc_ok(const Problem& p) {
    return p.items == 1 && p.K % 16 == 0 && p.N % 4 == 0 && p.M < (1LL << 31) && p.N < (1LL << 31) &&
           p.K < (1LL << 31);
}

size_t fp8_tc_workspace_bytes(const Problem& p) { return (size_t)(p.K * p.N); }

cudaError_t launch_fp8_simt(olc_dtype dt, const Problem& p, cudaStream_t s) {
    const int64_t tm = ceil_div(p.M, 64), tn = ceil_div(p.N, 64);
    const int64_t blocks = tm * tn * p.items;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    switch (dt) {
        case OLC_FLOAT8E4M3FN: f8::simt_kernel<0><<<(unsigned)blocks, 256, 0, s>>>(p, tm, tn); break;
        case OLC_FLOAT8E5M2: f8::simt_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(p, tm, tn); break;
        case OLC_FLOAT8E4M3FNUZ: f8::simt_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(p, tm, tn); break;
        case OLC_FLOAT8E5M2FNUZ: f8::simt_kernel<3><<<(unsigned)blocks, 256, 0, s>>>(p, tm, tn); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_fp8_transpose(const Problem& p, void* bt, cudaStream_t s) {
    const unsigned char* b = static_cast<const unsigned char*>(p.B);
    unsigned char* out = static_cast<unsigned char*>(bt);
    if (p.K <= 0 || p.N <= 0) return cudaSuccess;
    if (p.N % 16 == 0 && p.K % 16 == 0 && reinterpret_cast<uintptr_t>(b) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(out) % 16 == 0) {
        const int64_t ttn = ceil_div(p.N, f8::TT), ttk = ceil_div(p.K, f8::TT);
        if (ttn * ttk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        f8::transpose16_kernel<<<(unsigned)(ttn * ttk), 256, 0, s>>>(b, out, p.K, p.N, ttn);
    } else {
        const int64_t ttn = ceil_div(p.N, 64), ttk = ceil_div(p.K, 64);
        if (ttn * ttk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        f8::transpose_kernel<<<(unsigned)(ttn * ttk), 256, 0, s>>>(b, out, p.K, p.N, ttn);
    }
    return cudaGetLastError();
}

cudaError_t launch_fp8_tc(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                          cudaStream_t s, const void* bt_ready) {
    // the tensor cores take E4M3 and E5M2 (not the FNUZ encodings)
    if (!fp8_tc_ok(p) || (dt != OLC_FLOAT8E4M3FN && dt != OLC_FLOAT8E5M2)) return cudaErrorInvalidValue;
    const unsigned char* bt = static_cast<const unsigned char*>(bt_ready);
    if (!bt) {
        if (!ws.partials || ws.partial_bytes < fp8_tc_workspace_bytes(p)) return cudaErrorInvalidValue;
        const cudaError_t e = launch_fp8_transpose(p, ws.partials, s);
        if (e != cudaSuccess) return e;
        bt = static_cast<const unsigned char*>(ws.partials);
    }
    // CTA pairs (256 x 256 tiles, half of B per CTA) once the product holds
    // a pair tile; 128 x 256 tiles of one CTA otherwise (or when asked)
    if (p.M >= 256 && p.N >= 256 && p.variant != 1) return launch_pair_f8(dt, p, bt, sm_count, s);
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    if (!f8::encode_u8_2d(&ma, p.A, (uint64_t)p.K, (uint64_t)p.M, f8::BKB, f8::BM) ||
        !f8::encode_u8_2d(&mb, bt, (uint64_t)p.K, (uint64_t)p.N, f8::BKB, f8::BN))
        return cudaErrorInvalidValue;
    f8::Params q;
    std::memset(&q, 0, sizeof q);
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.tiles_m = ceil_div(p.M, f8::BM);
    q.tiles_n = ceil_div(p.N, f8::BN);
    q.total_tiles = q.tiles_m * q.tiles_n;
    q.k_blocks = ceil_div(p.K, f8::BKB);
    q.Y = static_cast<float*>(p.Y);
    q.err = device_error_word();
    q.fmt = dt == OLC_FLOAT8E4M3FN ? 0 : 1;
    q.epi = p.epi;
    const cudaError_t attr = set_smem_limit(reinterpret_cast<const void*>(f8::tc_kernel), f8::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const int64_t grid = min64(q.total_tiles, (int64_t)sm_count);
    f8::tc_kernel<<<(unsigned)grid, f8::THREADS, f8::SMEM_BYTES, s>>>(ma, mb, q);
    return cudaGetLastError();
}

}  // namespace olc

extern "C" uint32_t olc_debug_f8_instr_desc(int fmt, int m, int n) {
    return olc::f8::f8_instr_desc(fmt, m, n);
}
