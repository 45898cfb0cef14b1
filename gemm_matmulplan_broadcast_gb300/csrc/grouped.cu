// Grouped products: many independent rank-2 products Y_i = A_i @ B_i of
// different shapes in one persistent launch.
//
// "Gemm and MatMul Performance Roadmap": the batch-fusion row of its
// opportunity table (for hundreds of tiny or irregular products, one
// dispatch per product costs more than the product) and the GroupedGemm
// interface of its plan (small products scheduled together).  The plan
// numbers the 64 x 64 output tiles of all members consecutively (member i
// owns tiles [tile_begin_i, tile_begin_{i+1})); persistent blocks walk the
// tile numbers with a grid stride, find the member of a tile by binary search
// in the descriptor table, and compute the tile.  Members with an empty
// output own no tiles; K == 0 tiles are written as zeros.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"

namespace olc {
namespace {

constexpr int kGBM = 64, kGBN = 64, kGBK = 16, kGTM = 4, kGTN = 4;
constexpr int kGThreads = (kGBM / kGTM) * (kGBN / kGTN);   // 256

struct GDesc {
    int64_t m, n, k;
    int64_t tile_begin;     // first tile number of this member
    int64_t tiles_n;        // tiles along N
};

template <typename T>
__global__ void __launch_bounds__(kGThreads)
grouped_kernel(const GDesc* __restrict__ desc, int count, int64_t total_tiles,
               const void* const* __restrict__ Aptr, const void* const* __restrict__ Bptr,
               void* const* __restrict__ Yptr) {
    using acc_t = typename Num<T>::acc_t;
    constexpr int TX = kGBN / kGTN, TY = kGBM / kGTM;
    __shared__ acc_t As[kGBK][kGBM + 1];   // A tile, transposed: As[k][m]
    __shared__ acc_t Bs[kGBK][kGBN];
    const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;

    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        // member of this tile: the last i with tile_begin_i <= tile
        int lo = 0, hi = count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (desc[mid].tile_begin <= tile) lo = mid;
            else hi = mid - 1;
        }
        const GDesc d = desc[lo];
        const int64_t local = tile - d.tile_begin;
        const int64_t m0 = (local / d.tiles_n) * kGBM, n0 = (local % d.tiles_n) * kGBN;
        const int64_t M = d.m, N = d.n, K = d.k;
        const T* __restrict__ A = static_cast<const T*>(Aptr[lo]);
        const T* __restrict__ B = static_cast<const T*>(Bptr[lo]);
        T* __restrict__ Y = static_cast<T*>(Yptr[lo]);

        acc_t acc[kGTM][kGTN];
#pragma unroll
        for (int i = 0; i < kGTM; ++i)
#pragma unroll
            for (int j = 0; j < kGTN; ++j) acc[i][j] = acc_t(0);
        for (int64_t k0 = 0; k0 < K; k0 += kGBK) {
            __syncthreads();   // the previous step (or tile) is done with the tiles
            for (int e = threadIdx.x; e < kGBM * kGBK; e += kGThreads) {
                const int r = e / kGBK, c = e % kGBK;
                const int64_t gm = m0 + r, gk = k0 + c;
                As[c][r] = (gm < M && gk < K) ? Num<T>::to_acc(A[gm * K + gk]) : acc_t(0);
            }
            for (int e = threadIdx.x; e < kGBK * kGBN; e += kGThreads) {
                const int r = e / kGBN, c = e % kGBN;
                const int64_t gk = k0 + r, gn = n0 + c;
                Bs[r][c] = (gk < K && gn < N) ? Num<T>::to_acc(B[gk * N + gn]) : acc_t(0);
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < kGBK; ++kk) {
                acc_t a[kGTM], b[kGTN];
#pragma unroll
                for (int i = 0; i < kGTM; ++i) a[i] = As[kk][ty + i * TY];
#pragma unroll
                for (int j = 0; j < kGTN; ++j) b[j] = Bs[kk][tx + j * TX];
#pragma unroll
                for (int i = 0; i < kGTM; ++i)
#pragma unroll
                    for (int j = 0; j < kGTN; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < kGTM; ++i) {
            const int64_t gm = m0 + ty + i * TY;
            if (gm >= M) continue;
#pragma unroll
            for (int j = 0; j < kGTN; ++j) {
                const int64_t gn = n0 + tx + j * TX;
                if (gn < N) Y[gm * N + gn] = Num<T>::from_acc(acc[i][j]);
            }
        }
    }
}

}  // namespace
}  // namespace olc

struct olc_grouped_plan {
    olc_dtype dtype;
    int count;
    std::vector<olc::GDesc> desc;
    int64_t total_tiles;
    int device;                  // -1 until the descriptor table is on a device
    olc::GDesc* desc_dev;
    int sm_count;
};

namespace {

bool grouped_dtype_ok(olc_dtype dt) {
    return dt == OLC_FLOAT || dt == OLC_DOUBLE || dt == OLC_FLOAT16 || dt == OLC_BFLOAT16;
}

olc_status grouped_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return OLC_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? OLC_ERR_OOM : OLC_ERR_CUDA;
}

// descriptor table on the current device (once per plan)
olc_status grouped_bind(olc_grouped_plan* p) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return grouped_from_cuda(cudaErrorNoDevice);
    if (p->device >= 0) return cur == p->device ? OLC_OK : OLC_ERR_WRONG_DEVICE;
    void* mem = nullptr;
    const size_t bytes = sizeof(olc::GDesc) * (size_t)p->count;
    cudaError_t e = cudaMalloc(&mem, bytes);
    if (e == cudaSuccess) e = cudaMemcpy(mem, p->desc.data(), bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (mem) cudaFree(mem);
        return grouped_from_cuda(e);
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, cur) != cudaSuccess || sms <= 0)
        sms = 152;
    p->desc_dev = static_cast<olc::GDesc*>(mem);
    p->device = cur;
    p->sm_count = sms;
    return OLC_OK;
}

}  // namespace

extern "C" {

olc_status olc_grouped_plan_create(int count, const int64_t* m, const int64_t* n, const int64_t* k,
                                   olc_dtype dtype, olc_grouped_plan** out) {
    if (!out) return OLC_ERR_NULL;
    *out = nullptr;
    if (count <= 0) return OLC_ERR_INVALID;
    if (!m || !n || !k) return OLC_ERR_NULL;
    if (!grouped_dtype_ok(dtype)) return OLC_ERR_DTYPE;
    for (int i = 0; i < count; ++i)
        if (m[i] < 0 || n[i] < 0 || k[i] < 0) return OLC_ERR_NEGATIVE_DIM;
    olc_grouped_plan* p = new (std::nothrow) olc_grouped_plan;
    if (!p) return OLC_ERR_OOM;
    p->dtype = dtype;
    p->count = count;
    p->device = -1;
    p->desc_dev = nullptr;
    p->sm_count = 0;
    p->desc.resize((size_t)count);
    int64_t t = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t tm = olc::ceil_div(m[i], olc::kGBM), tn = olc::ceil_div(n[i], olc::kGBN);
        p->desc[i] = olc::GDesc{m[i], n[i], k[i], t, tn > 0 ? tn : 1};
        t += tm * tn;
    }
    p->total_tiles = t;
    *out = p;
    return OLC_OK;
}

void olc_grouped_plan_destroy(olc_grouped_plan* plan) {
    if (!plan) return;
    if (plan->desc_dev) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != plan->device) cudaSetDevice(plan->device);
        cudaFree(plan->desc_dev);
        if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    delete plan;
}

int64_t olc_grouped_plan_tiles(const olc_grouped_plan* plan) { return plan ? plan->total_tiles : -1; }

int olc_grouped_plan_count(const olc_grouped_plan* plan) { return plan ? plan->count : -1; }

olc_status olc_grouped_execute(const olc_grouped_plan* plan, const void* const* A, const void* const* B,
                               void* const* Y, void* stream) {
    if (!plan) return OLC_ERR_NULL;
    if (plan->total_tiles == 0) return OLC_OK;
    if (!A || !B || !Y) return OLC_ERR_NULL;
    olc_grouped_plan* p = const_cast<olc_grouped_plan*>(plan);
    olc_status st = grouped_bind(p);
    if (st != OLC_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t grid = olc::min64(plan->total_tiles, (int64_t)plan->sm_count * 4);
    cudaError_t e = olc::dispatch_dtype(plan->dtype, [&](auto tag) {
        using T = decltype(tag);
        olc::grouped_kernel<T><<<(unsigned)grid, olc::kGThreads, 0, s>>>(
            p->desc_dev, p->count, p->total_tiles, A, B, Y);
        return cudaGetLastError();
    });
    return grouped_from_cuda(e);
}

}  // extern "C"
