// SPLIT_K: tiny output, long reduction.
//
// "Gemm and MatMul Performance Roadmap", section "Parallel execution": when
// the whole M x N task grid cannot occupy the machine, K is partitioned into
// slices K0 | K1 | ..., each slice produces a partial product P_s with the
// same kernels, and a controlled reduction combines them
// (Y = P_0 + P_1 + ...).  Independent batches take priority over split-K (the
// plan only picks this path when tiles * batch items underfill the SMs).
//
// Here one launch does both passes.  Block (tile, s) accumulates its slice of
// K for a TM x TN output tile and writes the partial tile to the workspace;
// the last block to arrive for a tile (atomic counter) sums the partials in
// slice order s = 0, 1, ..., S-1 and writes the narrowed result.  The order of
// the final sum does not depend on which block arrives last, so the result is
// bit-reproducible run to run.
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace olc {

template <typename T>
struct SplitCfg {
    static constexpr int TM = 32, TN = 32, BK = 32;
    static constexpr int THREADS = 256;   // 2 x 2 outputs per thread
};

template <typename T>
__global__ void __launch_bounds__(256)
split_k_kernel(Problem p, int64_t tiles_m, int64_t tiles_n, int splits, int64_t kslice,
               Workspace ws) {
    using acc_t = typename Num<T>::acc_t;
    constexpr int TM = SplitCfg<T>::TM, TN = SplitCfg<T>::TN, BK = SplitCfg<T>::BK;
    __shared__ acc_t As[BK][TM + 1];
    __shared__ acc_t Bs[BK][TN];
    __shared__ unsigned int am_last;

    const int64_t tiles = tiles_m * tiles_n;
    const int64_t per_item = tiles * splits;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int s = (int)(rem / tiles);
    const int64_t t = rem % tiles;
    const int64_t m0 = (t / tiles_n) * TM, n0 = (t % tiles_n) * TN;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    T* __restrict__ Y = static_cast<T*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;
    const int64_t kb0 = (int64_t)s * kslice;
    const int64_t kb1 = min64(K, kb0 + kslice);

    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    acc_t acc[2][2] = {{acc_t(0), acc_t(0)}, {acc_t(0), acc_t(0)}};
    for (int64_t k0 = kb0; k0 < kb1; k0 += BK) {
        for (int e = threadIdx.x; e < TM * BK; e += 256) {
            const int r = e / BK, c = e % BK;
            const int64_t gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < kb1) ? Num<T>::to_acc(A[gm * K + gk]) : acc_t(0);
        }
        for (int e = threadIdx.x; e < BK * TN; e += 256) {
            const int r = e / TN, c = e % TN;
            const int64_t gk = k0 + r, gn = n0 + c;
            Bs[r][c] = (gk < kb1 && gn < N) ? Num<T>::to_acc(B[gk * N + gn]) : acc_t(0);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const acc_t a0 = As[kk][ty], a1 = As[kk][ty + 16];
            const acc_t b0 = Bs[kk][tx], b1 = Bs[kk][tx + 16];
            acc[0][0] = fma(a0, b0, acc[0][0]);
            acc[0][1] = fma(a0, b1, acc[0][1]);
            acc[1][0] = fma(a1, b0, acc[1][0]);
            acc[1][1] = fma(a1, b1, acc[1][1]);
        }
        __syncthreads();
    }

    constexpr int ENTRIES = TM * TN;
    acc_t* P = static_cast<acc_t*>(ws.partials);
    const int64_t tile_id = item * tiles + t;
    acc_t* mine = P + (tile_id * splits + s) * ENTRIES;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) mine[(ty + 16 * i) * TN + tx + 16 * j] = acc[i][j];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(ws.counters + tile_id, 1u);
        am_last = (prev == (unsigned int)splits - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!am_last) return;
    __threadfence();
    const acc_t* all = P + tile_id * splits * ENTRIES;
    for (int e = threadIdx.x; e < ENTRIES; e += 256) {
        // slice order 0, 1, ..., loads issued eight at a time
        acc_t v = acc_t(0);
        for (int q0 = 0; q0 < splits; q0 += 8) {
            acc_t t[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (q0 + j < splits) t[j] = __ldcg(all + (int64_t)(q0 + j) * ENTRIES + e);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (q0 + j < splits) v += t[j];
        }
        const int64_t gm = m0 + e / TN, gn = n0 + e % TN;
        if (gm < M && gn < N) Y[gm * N + gn] = Num<T>::from_acc(apply_epilogue<T>(p.epi, v, gm, gn, Y + gm * N + gn));
    }
    if (threadIdx.x == 0) ws.counters[tile_id] = 0u;
}

static int64_t acc_bytes(olc_dtype dt) { return dt == OLC_DOUBLE ? 8 : 4; }

int split_k_simt_pick(olc_dtype dt, const Problem& p, int sm_count) {
    (void)dt;
    if (p.split_hint > 0) return (int)min64(p.split_hint, max64(1, ceil_div(p.K, 32)));
    const int64_t tiles = ceil_div(p.M, 32) * ceil_div(p.N, 32) * p.items;
    // about two blocks per SM, each slice at least 256 long
    int64_t s = ceil_div(2LL * sm_count, tiles);
    const int64_t smax = max64(1, p.K / 256);
    if (s > smax) s = smax;
    if (s > 1024) s = 1024;
    return (int)max64(s, 1);
}

static size_t simt_partial_bytes(olc_dtype dt, const Problem& p, int splits) {
    const int64_t tiles = ceil_div(p.M, 32) * ceil_div(p.N, 32) * p.items;
    return (size_t)(tiles * splits * 32 * 32 * acc_bytes(dt));
}

static size_t simt_counter_count(const Problem& p) {
    return (size_t)(ceil_div(p.M, 32) * ceil_div(p.N, 32) * p.items);
}

cudaError_t launch_split_k_simt(olc_dtype dt, const Problem& p, int splits, const Workspace& ws,
                                cudaStream_t s) {
    if (!ws.partials || !ws.counters) return cudaErrorInvalidValue;
    const int64_t tm = ceil_div(p.M, 32), tn = ceil_div(p.N, 32);
    const int64_t kslice = ceil_div(ceil_div(p.K, splits), 32) * 32;
    const int64_t blocks = tm * tn * splits * p.items;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return dispatch_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        split_k_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(p, tm, tn, splits, kslice, ws);
        return cudaGetLastError();
    });
}

// FLOAT16 / BFLOAT16 with 16-byte row strides: the tensor-core kernel's
// split-K mode; everything else: the SIMT kernel above.
static bool split_on_tc(olc_dtype dt, const Problem& p) {
    return (dt == OLC_FLOAT16 || dt == OLC_BFLOAT16) && tc_shape_ok(dt, p.N, p.K);
}

// 8-bit float operands: the warp-MMA split-K (E4M3FN / E5M2, small outputs)
static bool is_f8(olc_dtype dt) {
    return dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2 || dt == OLC_FLOAT8E4M3FNUZ ||
           dt == OLC_FLOAT8E5M2FNUZ;
}

int split_k_pick(olc_dtype dt, const Problem& p, int sm_count) {
    if (is_f8(dt)) return f8_split_k_pick(p, sm_count);
    return split_on_tc(dt, p) ? tc_split_pick(p, sm_count) : split_k_simt_pick(dt, p, sm_count);
}

size_t split_k_partial_bytes(olc_dtype dt, const Problem& p, int splits, int sm_count) {
    if (is_f8(dt)) return splits > 1 ? f8_split_k_partial_bytes(p, splits) : 0;
    return split_on_tc(dt, p) ? tc_split_partial_bytes(p, sm_count)
                              : simt_partial_bytes(dt, p, splits);
}

size_t split_k_counter_count(olc_dtype dt, const Problem& p, int splits, int sm_count) {
    if (is_f8(dt)) return splits > 1 ? f8_split_k_counter_count(p, splits) : 0;
    return split_on_tc(dt, p) ? tc_split_counter_count(p, sm_count) : simt_counter_count(p);
}

cudaError_t launch_split_k(olc_dtype dt, const Problem& p, int splits, int sm_count,
                           const Workspace& ws, cudaStream_t s) {
    if (is_f8(dt)) return launch_f8_split_k(dt, p, splits, ws, s);
    if (split_on_tc(dt, p)) return launch_tc_split(dt, p, sm_count, ws, s);
    return launch_split_k_simt(dt, p, splits, ws, s);
}

}  // namespace olc

// ===========================================================================
// Allocation-free split-K: the same kernel, with its partial tiles and arrival
// counters in a file-scope device array instead of a cudaMalloc'd workspace,
// for callers that must not allocate device memory while they run.

namespace olc {
namespace {

constexpr size_t kStaticScratchBytes = OLC_SPLIT_K_STATIC_SCRATCH_BYTES;
constexpr size_t kStaticCounterBytes = 16 * 1024;   // 4096 counters
constexpr size_t kStaticPartialBytes = kStaticScratchBytes - kStaticCounterBytes;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_split_k_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_split_k_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace olc

extern "C" olc_status olc_matmul_split_k_static(olc_dtype dtype, const void* A, const void* B,
                                                void* Y, int64_t M, int64_t N, int64_t K,
                                                void* stream) {
    using namespace olc;
    if (dtype != OLC_FLOAT && dtype != OLC_DOUBLE && dtype != OLC_FLOAT16 &&
        dtype != OLC_BFLOAT16)
        return OLC_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0) return OLC_ERR_NEGATIVE_DIM;
    if (M == 0 || N == 0) return OLC_OK;
    if (!Y) return OLC_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t eb = dtype == OLC_DOUBLE ? 8 : dtype == OLC_FLOAT ? 4 : 2;
    if (K == 0) {
        return launch_zero_fill(Y, M * N * eb, s) == cudaSuccess ? OLC_OK : OLC_ERR_CUDA;
    }
    if (!A || !B) return OLC_ERR_NULL;

    Problem p;
    std::memset(&p, 0, sizeof p);
    p.A = A;
    p.B = B;
    p.Y = Y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.items = 1;
    p.split_hint = 0;
    const int64_t tiles = ceil_div(M, 32) * ceil_div(N, 32);
    const int64_t tile_bytes = 32 * 32 * acc_bytes(dtype);
    if (tiles * (int64_t)sizeof(unsigned int) > (int64_t)kStaticCounterBytes ||
        tiles * tile_bytes > (int64_t)kStaticPartialBytes)
        return OLC_ERR_SCRATCH_LIMIT;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    // the array's address and the SM count are the current device's: a
    // stream of another device would get an address of the wrong context
    if (s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread) {
        int sdev = -1;
        if (cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
            cudaGetLastError();
            return OLC_ERR_CUDA;
        }
        if (sdev != dev) return OLC_ERR_WRONG_DEVICE;
    }
    int splits = split_k_simt_pick(dtype, p, sms);
    const int64_t fit = (int64_t)kStaticPartialBytes / (tiles * tile_bytes);
    if (splits > fit) splits = (int)fit;
    if (splits < 1) splits = 1;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    Workspace ws;
    ws.counters = static_cast<unsigned int*>(base);
    ws.counter_count = (size_t)tiles;
    ws.partials = static_cast<unsigned char*>(base) + kStaticCounterBytes;
    ws.partial_bytes = (size_t)(tiles * splits * tile_bytes);
    // the counters must start at zero for this launch, whatever an earlier
    // call left behind
    if (cudaMemsetAsync(ws.counters, 0, (size_t)tiles * sizeof(unsigned int), s) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    if (launch_split_k_simt(dtype, p, splits, ws, s) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    return OLC_OK;
}
