// SIMT tile kernels: DIRECT (any shape, any alignment) and the first
// GENERAL_SIMT.  Also the zero-fill kernel and the device error word.
//
// "MatMul Kernel Design", section "Types and algorithm selection": direct
// execution for small natural-layout reductions.  Operands are read in their
// natural row-major layout (no packing pass); each block owns a BM x BN tile
// of one batch item's output, stages BK-deep slices of A (transposed) and B
// in shared memory already widened to the accumulator type, and each thread
// keeps a TM x TN register tile.  Every output sums its K products in
// ascending k with fused multiply-adds in the accumulator type (float32 for
// FLOAT/FLOAT16/BFLOAT16, float64 for DOUBLE).
#include <mutex>

#include "common.cuh"

namespace olc {

__device__ unsigned int g_device_error = 0;

// Looked up once per device (not on every launch, so launches can be
// captured into CUDA graphs without runtime symbol queries).
unsigned int* device_error_word() {
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = ptr;
    }
    return static_cast<unsigned int*>(cache[dev]);
}

cudaError_t read_and_clear_device_error(unsigned int* value, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_device_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*value != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

// ---------------------------------------------------------------------------
// zero fill (K == 0): 16-byte stores where the pointer allows, bytes otherwise

__global__ void zero_fill_kernel(unsigned char* y, int64_t bytes) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uintptr_t base = reinterpret_cast<uintptr_t>(y);
    const int64_t head = (int64_t)((16 - (base & 15)) & 15) < bytes ? (int64_t)((16 - (base & 15)) & 15) : bytes;
    const int64_t body = (bytes - head) / 16;
    for (int64_t t = i; t < head; t += stride) y[t] = 0;
    uint4* v = reinterpret_cast<uint4*>(y + head);
    for (int64_t t = i; t < body; t += stride) v[t] = make_uint4(0, 0, 0, 0);
    for (int64_t t = head + body * 16 + i; t < bytes; t += stride) y[t] = 0;
}

cudaError_t launch_zero_fill(void* Y, int64_t bytes, cudaStream_t stream) {
    if (bytes <= 0) return cudaSuccess;
    int64_t blocks = ceil_div(bytes / 16 + 1, 256);
    if (blocks > 4096) blocks = 4096;
    zero_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<unsigned char*>(Y), bytes);
    return cudaGetLastError();
}

// Gemm with K == 0: Y = beta * C (or 0 without C), elementwise
template <typename T>
__global__ void epilogue_fill_kernel(Problem p) {
    using acc_t = typename Num<T>::acc_t;
    const int64_t n = p.M * p.N;
    T* Y = static_cast<T*>(p.Y);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x)
        Y[e] = Num<T>::from_acc(apply_epilogue<T>(p.epi, acc_t(0), e / p.N, e % p.N, Y + e));
}

cudaError_t launch_epilogue_fill(olc_dtype dt, const Problem& p, cudaStream_t stream) {
    const int64_t n = p.M * p.N;
    if (n <= 0) return cudaSuccess;
    int64_t blocks = ceil_div(n, 256);
    if (blocks > 4096) blocks = 4096;
    return dispatch_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        epilogue_fill_kernel<T><<<(unsigned)blocks, 256, 0, stream>>>(p);
        return cudaGetLastError();
    });
}

// ---------------------------------------------------------------------------
// the tile kernel

template <typename T, int BM, int BN, int BK, int TM, int TN>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
tile_gemm_kernel(Problem p, int64_t tiles_m, int64_t tiles_n) {
    using acc_t = typename Num<T>::acc_t;
    constexpr int TX = BN / TN;          // threads along N
    constexpr int TY = BM / TM;          // threads along M
    constexpr int NT = TX * TY;
    __shared__ acc_t As[BK][BM + 1];     // A tile, transposed: As[k][m]
    __shared__ acc_t Bs[BK][BN];

    const int64_t per_item = tiles_m * tiles_n;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int64_t m0 = (rem / tiles_n) * BM;
    const int64_t n0 = (rem % tiles_n) * BN;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    T* __restrict__ Y = static_cast<T*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;

    const int tx = threadIdx.x % TX;
    const int ty = threadIdx.x / TX;
    // launched with programmatic dependent launch: wait for the previous
    // kernel in the stream before touching global memory; the next launch
    // is released once this block's products are done (released at the
    // start, the next kernel's blocks would hold SM resources through all
    // of this one)
    grid_dependency_wait();
    acc_t acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = acc_t(0);

    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        for (int e = threadIdx.x; e < BM * BK; e += NT) {
            const int r = e / BK, c = e % BK;
            const int64_t gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K)
                           ? Num<T>::to_acc(p.a_trans ? A[gk * M + gm] : A[gm * K + gk])
                           : acc_t(0);
        }
        for (int e = threadIdx.x; e < BK * BN; e += NT) {
            const int r = e / BN, c = e % BN;
            const int64_t gk = k0 + r, gn = n0 + c;
            Bs[r][c] = (gk < K && gn < N)
                           ? Num<T>::to_acc(p.b_trans ? B[gn * K + gk] : B[gk * N + gn])
                           : acc_t(0);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            acc_t a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[kk][ty + i * TY];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = Bs[kk][tx + j * TX];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    grid_launch_dependents();
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + ty + i * TY;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t gn = n0 + tx + j * TX;
            if (gn < N) Y[gm * N + gn] = Num<T>::from_acc(apply_epilogue<T>(p.epi, acc[i][j], gm, gn, Y + gm * N + gn));
        }
    }
}

template <typename T, int BM, int BN, int BK, int TM, int TN>
static cudaError_t launch_tile(const Problem& p, cudaStream_t stream) {
    const int64_t tm = ceil_div(p.M, BM), tn = ceil_div(p.N, BN);
    const int64_t blocks = tm * tn * p.items;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(tile_gemm_kernel<T, BM, BN, BK, TM, TN>, dim3((unsigned)blocks),
                      dim3((BM / TM) * (BN / TN)), 0, stream, p, tm, tn);
}

// ---------------------------------------------------------------------------
// DIRECT for small FLOAT / DOUBLE products: the whole K range at once.
//
// Small products are latency-bound: the slice loop above pays one global
// round trip per 16-deep slice.  Here a block issues every element copy of
// its 32 x K strip of A and K x 32 strip of B at once (cp.async, one element
// each, so any alignment and any K), waits once, and then multiplies from
// shared memory; each thread sums its 2 x 2 outputs over k ascending with
// fused multiply-adds, as the slice kernel does.  K is bounded so that both
// strips fit in 64 KiB of shared memory (K <= 256 for FLOAT, 128 for
// DOUBLE); operands stored as given (no Gemm transposes).

template <typename T>
constexpr int wholek_max_k() { return sizeof(T) == 4 ? 256 : 128; }

__device__ __forceinline__ void cp_async_elem(void* smem, const void* gmem, int bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    if (bytes == 4)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(gmem) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(256) wholek_kernel(Problem p, int64_t tiles_m, int64_t tiles_n) {
    extern __shared__ __align__(16) unsigned char wk_smem[];
    const int64_t K = p.K;
    const int ks = (int)K + 1;                 // A row stride: odd, so the two rows a warp reads differ in bank
    T* As = reinterpret_cast<T*>(wk_smem);     // [32][ks]
    T* Bs = As + 32 * ks;                      // [K][32]

    const int64_t per_item = tiles_m * tiles_n;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int64_t m0 = (rem / tiles_n) * 32;
    const int64_t n0 = (rem % tiles_n) * 32;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    T* __restrict__ Y = static_cast<T*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependency_wait();                    // programmatic dependent launch, as above

    // A rows m0 + r (r = warp, warp + 8, ...), lanes along k; B rows k
    // (k = warp, warp + 8, ...), lanes along n.  Outside the product: zeros.
    for (int r = warp; r < 32; r += 8) {
        const bool ok = m0 + r < M;
        const T* src = A + (m0 + r) * K;
        for (int k = lane; k < (int)K; k += 32) {
            if (ok) cp_async_elem(As + r * ks + k, src + k, (int)sizeof(T));
            else As[r * ks + k] = T(0);
        }
    }
    const bool col_ok = n0 + lane < N;
    for (int k = warp; k < (int)K; k += 8) {
        if (col_ok) cp_async_elem(Bs + k * 32 + lane, B + (int64_t)k * N + n0 + lane, (int)sizeof(T));
        else Bs[k * 32 + lane] = T(0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    T c00 = T(0), c01 = T(0), c10 = T(0), c11 = T(0);
    const T* a0p = As + ty * ks;
    const T* a1p = As + (ty + 16) * ks;
#pragma unroll 4
    for (int k = 0; k < (int)K; ++k) {
        const T a0 = a0p[k], a1 = a1p[k];
        const T b0 = Bs[k * 32 + tx], b1 = Bs[k * 32 + tx + 16];
        c00 = fma(a0, b0, c00);
        c01 = fma(a0, b1, c01);
        c10 = fma(a1, b0, c10);
        c11 = fma(a1, b1, c11);
    }
    grid_launch_dependents();
    const T c[2][2] = {{c00, c01}, {c10, c11}};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int64_t gm = m0 + ty + 16 * i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t gn = n0 + tx + 16 * j;
            if (gn < N) Y[gm * N + gn] = apply_epilogue<T>(p.epi, c[i][j], gm, gn, Y + gm * N + gn);
        }
    }
}

bool direct_wholek_ok(olc_dtype dt, const Problem& p) {
    if (p.a_trans || p.b_trans || p.K < 1) return false;
    if (dt == OLC_FLOAT) return p.K <= wholek_max_k<float>();
    if (dt == OLC_DOUBLE) return p.K <= wholek_max_k<double>();
    return false;
}

template <typename T>
static cudaError_t launch_wholek(const Problem& p, cudaStream_t stream) {
    const int64_t tm = ceil_div(p.M, 32), tn = ceil_div(p.N, 32);
    const int64_t blocks = tm * tn * p.items;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)(32 * (p.K + 1) + p.K * 32) * sizeof(T);
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(wholek_kernel<T>),
                                         (int)((32 * (wholek_max_k<T>() + 1) + wholek_max_k<T>() * 32) * sizeof(T)));
    if (e != cudaSuccess) return e;
    return launch_pdl(wholek_kernel<T>, dim3((unsigned)blocks), dim3(256), smem, stream, p, tm, tn);
}

cudaError_t launch_direct(olc_dtype dt, const Problem& p, cudaStream_t stream) {
    if (direct_wholek_ok(dt, p))
        return dt == OLC_FLOAT ? launch_wholek<float>(p, stream) : launch_wholek<double>(p, stream);
    return dispatch_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return launch_tile<T, 32, 32, 16, 2, 2>(p, stream);
    });
}

cudaError_t launch_general_simt_generic(olc_dtype dt, const Problem& p, cudaStream_t stream) {
    return dispatch_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return launch_tile<T, 64, 64, 16, 4, 4>(p, stream);
    });
}

}  // namespace olc

namespace olc {

// ---------------------------------------------------------------------------
// GENERAL_SIMT fast path: FP32 FFMA / FP64 DFMA register tiles
//
// Block tile BM x BN, BK-deep slices, 256 threads in a 16 x 16 grid; each
// thread owns a TM x TN register tile split into two halves in each
// direction (rows ty*TM/2 + i and BM/2 + ty*TM/2 + i, the same for columns),
// so that the shared-memory reads of a warp are broadcasts (A) or one
// contiguous run (B).  A's slice is stored transposed (As[k][m]) so a thread
// reads its rows as 16-byte vectors.  The next slice is loaded from global
// memory into registers while the current one is multiplied (two
// shared-memory buffers, one barrier per slice).  Every output sums its K
// products in ascending k with fused multiply-adds in the element type.
// Needs K and N multiples of the 16-byte vector width and 16-byte aligned
// operands; other shapes take the generic tile kernel above.

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    using type = float4;
    static constexpr int W = 4;
};
template <>
struct Vec<double> {
    using type = double2;
    static constexpr int W = 2;
};

constexpr int SIMT_GROUP_M = 16;

template <typename T, int BM, int BN, int BK, int TM, int TN, bool AT, bool BT>
__global__ void __launch_bounds__(256, 2)
simt_fast_kernel(Problem p, int64_t tiles_m, int64_t tiles_n, int splits, int64_t k_slice,
                 T* __restrict__ part, unsigned int* __restrict__ cnt) {
    using V = typename Vec<T>::type;
    constexpr int W = Vec<T>::W;
    constexpr int PAD = W;
    constexpr int HM = TM / 2, HN = TN / 2;
    constexpr bool PAIRED = sizeof(T) == 4;      // FP32: accumulate with f32x2 FMAs
    static_assert(BM == 16 * TM && BN == 16 * TN, "16 x 16 threads");
    static_assert(HM % W == 0 && HN % W == 0, "half tiles are whole vectors");
    constexpr int AV = (BM * BK) / W / 256;      // A vectors per thread per slice
    constexpr int BV = (BK * BN) / W / 256;      // B vectors per thread per slice
    static_assert(AV * W * 256 == BM * BK && BV * W * 256 == BK * BN, "whole vectors per thread");
    __shared__ __align__(16) T As[2][BK][BM + PAD];
    __shared__ __align__(16) T Bs[2][BK][BN];

    // K slice (splits > 1: slice s covers [s * k_slice, (s + 1) * k_slice),
    // k_slice a multiple of BK) and tile of this block
    const int64_t per_item = tiles_m * tiles_n;
    const int64_t all_tiles = per_item * p.items;
    const int slice = (int)(blockIdx.x / all_tiles);
    const int64_t tile_id = blockIdx.x % all_tiles;
    const int64_t item = tile_id / per_item;
    const int64_t rem = tile_id % per_item;
    // tile raster in groups of SIMT_GROUP_M row blocks, column-major inside a
    // group: the blocks resident at one time share a few A row strips and B
    // column strips, so L2 serves most re-reads instead of DRAM
    const int64_t span = (int64_t)SIMT_GROUP_M * tiles_n;
    const int64_t first = (rem / span) * SIMT_GROUP_M;
    const int64_t gm = min64(tiles_m - first, (int64_t)SIMT_GROUP_M);
    const int64_t in = rem % span;
    const int64_t m0 = (first + in % gm) * BM;
    const int64_t n0 = (in / gm) * BN;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    T* __restrict__ Y = static_cast<T*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;
    const int64_t k_begin = splits > 1 ? (int64_t)slice * k_slice : 0;
    const int64_t k_end = splits > 1 ? min64(K, k_begin + k_slice) : K;

    const int t = threadIdx.x;
    const int tx = t % 16, ty = t / 16;
    constexpr int AVR = BK / W;                   // vectors per A row slice
    constexpr int BVR = BN / W;                   // vectors per B row

    // A stored [M, K]: vectors along K, stored transposed into As[k][m];
    // A stored [K, M] (Gemm transA): vectors along M, stored as they are.
    // B stored [K, N]: vectors along N; B stored [N, K] (transB): vectors
    // along K, stored transposed into Bs[k][n].
    constexpr int AMR = BM / W;                   // vectors per A k-row (transposed A)
    constexpr int BKR = BK / W;                   // vectors per B n-row (transposed B)
    constexpr bool at = AT, bt = BT;
    auto load_a = [&](int64_t k0, V (&v)[AV]) {
#pragma unroll
        for (int q = 0; q < AV; ++q) {
            const int e = t + q * 256;
            if (!at) {
                const int64_t row = m0 + e / AVR, k = k0 + (e % AVR) * W;
                if (row < M && k < K) v[q] = *reinterpret_cast<const V*>(A + row * K + k);
                else v[q] = V{};
            } else {
                const int64_t k = k0 + e / AMR, row = m0 + (e % AMR) * W;
                if (k < K && row < M) v[q] = *reinterpret_cast<const V*>(A + k * M + row);
                else v[q] = V{};
            }
        }
    };
    auto load_b = [&](int64_t k0, V (&v)[BV]) {
#pragma unroll
        for (int q = 0; q < BV; ++q) {
            const int e = t + q * 256;
            if (!bt) {
                const int64_t k = k0 + e / BVR, col = n0 + (e % BVR) * W;
                if (k < K && col < N) v[q] = *reinterpret_cast<const V*>(B + k * N + col);
                else v[q] = V{};
            } else {
                const int64_t col = n0 + e / BKR, k = k0 + (e % BKR) * W;
                if (col < N && k < K) v[q] = *reinterpret_cast<const V*>(B + col * K + k);
                else v[q] = V{};
            }
        }
    };
    auto store_stage = [&](int buf, const V (&va)[AV], const V (&vb)[BV]) {
#pragma unroll
        for (int q = 0; q < AV; ++q) {
            const int e = t + q * 256;
            if (!at) {
                const int row = e / AVR, kk = (e % AVR) * W;
                const T* ae = reinterpret_cast<const T*>(&va[q]);
#pragma unroll
                for (int i = 0; i < W; ++i) As[buf][kk + i][row] = ae[i];
            } else {
                *reinterpret_cast<V*>(&As[buf][e / AMR][(e % AMR) * W]) = va[q];
            }
        }
#pragma unroll
        for (int q = 0; q < BV; ++q) {
            const int e = t + q * 256;
            if (!bt) {
                *reinterpret_cast<V*>(&Bs[buf][e / BVR][(e % BVR) * W]) = vb[q];
            } else {
                const int col = e / BKR, kk = (e % BKR) * W;
                const T* be = reinterpret_cast<const T*>(&vb[q]);
#pragma unroll
                for (int i = 0; i < W; ++i) Bs[buf][kk + i][col] = be[i];
            }
        }
    };

    T acc[TM][TN];
    unsigned long long acc2[TM][TN / 2];
#pragma unroll
    for (int i = 0; i < TM; ++i) {
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = T(0);
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc2[i][j] = 0ull;   // +0.0f, +0.0f
    }

    V va[AV], vb[BV];
    load_a(k_begin, va);
    load_b(k_begin, vb);
    store_stage(0, va, vb);
    __syncthreads();
    int buf = 0;
    for (int64_t k0 = k_begin; k0 < k_end; k0 += BK) {
        const bool more = k0 + BK < k_end;
        if (more) {
            load_a(k0 + BK, va);
            load_b(k0 + BK, vb);
        }
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            T a[TM], b[TN];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int q = 0; q < HM / W; ++q) {
                    const V v = *reinterpret_cast<const V*>(&As[buf][kk][h * (BM / 2) + ty * HM + q * W]);
                    const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
                    for (int i = 0; i < W; ++i) a[h * HM + q * W + i] = e[i];
                }
#pragma unroll
                for (int q = 0; q < HN / W; ++q) {
                    const V v = *reinterpret_cast<const V*>(&Bs[buf][kk][h * (BN / 2) + tx * HN + q * W]);
                    const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
                    for (int i = 0; i < W; ++i) b[h * HN + q * W + i] = e[i];
                }
            }
            if constexpr (PAIRED) {
                unsigned long long b2[TN / 2];
#pragma unroll
                for (int j = 0; j < TN / 2; ++j) b2[j] = pack_f2(b[2 * j], b[2 * j + 1]);
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const unsigned long long a2 = pack_f2(a[i], a[i]);
#pragma unroll
                    for (int j = 0; j < TN / 2; ++j) fma_f2(acc2[i][j], a2, b2[j]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
            }
        }
        if (more) {
            store_stage(buf ^ 1, va, vb);
            __syncthreads();
            buf ^= 1;
        }
    }
    if constexpr (PAIRED) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) {
                float lo, hi;
                unpack_f2(acc2[i][j], lo, hi);
                acc[i][2 * j] = lo;
                acc[i][2 * j + 1] = hi;
            }
    }

    if (splits > 1) {
        // this slice's partial tile, in the thread's own register order
        constexpr int F = TM * TN;
        T* mine = part + ((int64_t)tile_id * splits + slice) * (256 * F) + (int64_t)t * F;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; j += W) {
                V v;
                T* e = reinterpret_cast<T*>(&v);
#pragma unroll
                for (int q = 0; q < W; ++q) e[q] = acc[i][j + q];
                *reinterpret_cast<V*>(mine + i * TN + j) = v;
            }
        __threadfence();
        __syncthreads();
        __shared__ int last;
        if (t == 0) {
            const unsigned int prev = atomicAdd(cnt + tile_id, 1u);
            last = prev == (unsigned int)splits - 1 ? 1 : 0;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
        // the last slice to finish sums the slices in slice order
        const T* first = part + (int64_t)tile_id * splits * (256 * F) + (int64_t)t * F;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = T(0);
        for (int s2 = 0; s2 < splits; ++s2) {
            const T* src = first + (int64_t)s2 * (256 * F);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; j += W) {
                    const V v = __ldcg(reinterpret_cast<const V*>(src + i * TN + j));
                    const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
                    for (int q = 0; q < W; ++q) acc[i][j + q] += e[q];
                }
        }
        if (t == 0) cnt[tile_id] = 0u;
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + (i / HM) * (BM / 2) + ty * HM + (i % HM);
        if (gm >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int q = 0; q < HN / W; ++q) {
                const int64_t gn = n0 + h * (BN / 2) + tx * HN + q * W;
                if (gn < N) {   // N is a multiple of W: the whole vector is inside
                    V v;
                    T* e = reinterpret_cast<T*>(&v);
#pragma unroll
                    for (int j = 0; j < W; ++j)
                        e[j] = apply_epilogue<T>(p.epi, acc[i][h * HN + q * W + j], gm, gn + j,
                                                        Y + gm * N + gn + j);
                    *reinterpret_cast<V*>(Y + gm * N + gn) = v;
                }
            }
        }
    }
}

// K slice length for `splits` slices: a multiple of BK, so that slice
// boundaries fall on the kernel's BK-deep steps
static int64_t simt_k_slice(int64_t K, int splits, int bk) {
    return ceil_div(ceil_div(K, (int64_t)splits), (int64_t)bk) * bk;
}

template <typename T, int BM, int BN, int BK, int TM, int TN>
static cudaError_t launch_fast(const Problem& p, cudaStream_t stream, int splits, const Workspace* ws) {
    const int64_t tm = ceil_div(p.M, BM), tn = ceil_div(p.N, BN);
    const int64_t tiles = tm * tn * p.items;
    if (tiles <= 0) return cudaSuccess;
    int64_t k_slice = p.K;
    T* part = nullptr;
    unsigned int* cnt = nullptr;
    if (splits > 1) {
        k_slice = simt_k_slice(p.K, splits, BK);
        splits = (int)ceil_div(p.K, k_slice);          // non-empty slices
    }
    if (splits > 1) {
        const size_t need = (size_t)tiles * splits * BM * BN * sizeof(T);
        if (!ws || !ws->partials || ws->partial_bytes < need || !ws->counters ||
            ws->counter_count < (size_t)tiles)
            return cudaErrorInvalidValue;
        part = static_cast<T*>(ws->partials);
        cnt = ws->counters;
    } else {
        splits = 1;
        k_slice = p.K;
    }
    const int64_t blocks = tiles * splits;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const unsigned g = (unsigned)blocks;
    if (!p.a_trans && !p.b_trans)
        simt_fast_kernel<T, BM, BN, BK, TM, TN, false, false>
            <<<g, 256, 0, stream>>>(p, tm, tn, splits, k_slice, part, cnt);
    else if (p.a_trans && !p.b_trans)
        simt_fast_kernel<T, BM, BN, BK, TM, TN, true, false>
            <<<g, 256, 0, stream>>>(p, tm, tn, splits, k_slice, part, cnt);
    else if (!p.a_trans && p.b_trans)
        simt_fast_kernel<T, BM, BN, BK, TM, TN, false, true>
            <<<g, 256, 0, stream>>>(p, tm, tn, splits, k_slice, part, cnt);
    else
        simt_fast_kernel<T, BM, BN, BK, TM, TN, true, true>
            <<<g, 256, 0, stream>>>(p, tm, tn, splits, k_slice, part, cnt);
    return cudaGetLastError();
}

bool general_simt_fast_ok(olc_dtype dt, int64_t N, int64_t K) {
    if (dt == OLC_FLOAT) return N % 4 == 0 && K % 4 == 0;
    if (dt == OLC_DOUBLE) return N % 2 == 0 && K % 2 == 0;
    return false;
}

static bool fast_shape_ok(olc_dtype dt, const Problem& p) {
    const int64_t w = dt == OLC_FLOAT ? 4 : 2;
    return general_simt_fast_ok(dt, p.N, p.K) && (!p.a_trans || p.M % w == 0);
}

static bool aligned_items(const Problem& p, int64_t elem) {
    if ((reinterpret_cast<uintptr_t>(p.A) | reinterpret_cast<uintptr_t>(p.B) |
         reinterpret_cast<uintptr_t>(p.Y)) & 15)
        return false;
    for (int d = 0; d < p.map.rank; ++d)
        if (((p.map.a_stride[d] | p.map.b_stride[d]) * elem) % 16 != 0) return false;
    return ((p.M * p.N) * elem) % 16 == 0;
}

cudaError_t launch_general_simt_fast(olc_dtype dt, const Problem& p, cudaStream_t stream, int splits,
                                     const Workspace* ws) {
    if (!fast_shape_ok(dt, p)) return launch_general_simt_generic(dt, p, stream);
    if (dt == OLC_FLOAT && aligned_items(p, 4))
        return launch_fast<float, 128, 128, 16, 8, 8>(p, stream, splits, ws);
    if (dt == OLC_DOUBLE && aligned_items(p, 8))
        return launch_fast<double, 64, 64, 8, 4, 4>(p, stream, 1, nullptr);
    return launch_general_simt_generic(dt, p, stream);
}

// FLOAT products whose 128 x 128 tiles leave SMs idle: with fewer tiles than
// SMs, enough K slices to give each SM about two blocks; with one partial
// wave of two blocks per SM, 4 slices (measured on 256-tile products: +8 %;
// 2 or 3 slices: no gain); slices of at least 128 (8 steps of 16)
int general_simt_pick_split(olc_dtype dt, const Problem& p, int sm_count) {
    if (dt != OLC_FLOAT || !fast_shape_ok(dt, p) || p.split_hint == 1) return 1;
    const int64_t tiles = ceil_div(p.M, 128) * ceil_div(p.N, 128) * p.items;
    if (tiles <= 0 || p.K <= 0) return 1;
    int64_t s = 1;
    if (p.split_hint > 1) s = p.split_hint;
    else if (tiles < sm_count) s = (2 * sm_count) / tiles;
    else if (tiles < 2 * sm_count) s = 4;
    s = min64(s, max64(1, p.K / 128));
    s = min64(s, 16);
    if (s < 2) return 1;
    return (int)ceil_div(p.K, simt_k_slice(p.K, (int)s, 16));   // non-empty slices
}

size_t general_simt_partial_bytes(olc_dtype dt, const Problem& p, int splits) {
    if (splits < 2 || dt != OLC_FLOAT) return 0;
    return (size_t)(ceil_div(p.M, 128) * ceil_div(p.N, 128) * p.items) * splits * 128 * 128 * 4;
}

size_t general_simt_counter_count(olc_dtype dt, const Problem& p, int splits) {
    if (splits < 2 || dt != OLC_FLOAT) return 0;
    return (size_t)(ceil_div(p.M, 128) * ceil_div(p.N, 128) * p.items);
}

}  // namespace olc
