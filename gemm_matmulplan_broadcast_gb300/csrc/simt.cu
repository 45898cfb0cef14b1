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
#include "common.cuh"

namespace olc {

__device__ unsigned int g_device_error = 0;

unsigned int* device_error_word() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return static_cast<unsigned int*>(ptr);
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
    acc_t acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = acc_t(0);

    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        for (int e = threadIdx.x; e < BM * BK; e += NT) {
            const int r = e / BK, c = e % BK;
            const int64_t gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K) ? Num<T>::to_acc(A[gm * K + gk]) : acc_t(0);
        }
        for (int e = threadIdx.x; e < BK * BN; e += NT) {
            const int r = e / BN, c = e % BN;
            const int64_t gk = k0 + r, gn = n0 + c;
            Bs[r][c] = (gk < K && gn < N) ? Num<T>::to_acc(B[gk * N + gn]) : acc_t(0);
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
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + ty + i * TY;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t gn = n0 + tx + j * TX;
            if (gn < N) Y[gm * N + gn] = Num<T>::from_acc(acc[i][j]);
        }
    }
}

template <typename T, int BM, int BN, int BK, int TM, int TN>
static cudaError_t launch_tile(const Problem& p, cudaStream_t stream) {
    const int64_t tm = ceil_div(p.M, BM), tn = ceil_div(p.N, BN);
    const int64_t blocks = tm * tn * p.items;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    tile_gemm_kernel<T, BM, BN, BK, TM, TN>
        <<<(unsigned)blocks, (BM / TM) * (BN / TN), 0, stream>>>(p, tm, tn);
    return cudaGetLastError();
}

cudaError_t launch_direct(olc_dtype dt, const Problem& p, cudaStream_t stream) {
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
bool general_simt_fast_ok(olc_dtype dt, int64_t N, int64_t K) {
    (void)dt; (void)N; (void)K;
    return false;
}
cudaError_t launch_general_simt_fast(olc_dtype dt, const Problem& p, cudaStream_t stream) {
    return launch_general_simt_generic(dt, p, stream);
}
}  // namespace olc
