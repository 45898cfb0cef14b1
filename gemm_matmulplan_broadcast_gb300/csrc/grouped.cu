// Grouped products: many independent rank-2 products Y_i = A_i @ B_i of
// different shapes in one persistent launch.
//
// "Gemm and MatMul Performance Roadmap": the batch-fusion row of its
// opportunity table (for hundreds of tiny or irregular products, one
// dispatch per product costs more than the product) and the GroupedGemm
// interface of its plan (small products scheduled together).  The plan
// numbers the 64 x 64 output tiles of all members consecutively (member i
// owns tiles [tile_begin_i, tile_begin_{i+1})) and keeps, next to the
// descriptor table, the owning member of every tile; persistent blocks walk
// the tile numbers with a grid stride, read the tile's member (one load),
// and compute the tile.  Members with an empty
// output own no tiles; K == 0 tiles are written as zeros.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>
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
grouped_kernel(const GDesc* __restrict__ desc, const int* __restrict__ owner, int64_t total_tiles,
               const void* const* __restrict__ Aptr, const void* const* __restrict__ Bptr,
               void* const* __restrict__ Yptr) {
    using acc_t = typename Num<T>::acc_t;
    constexpr int TX = kGBN / kGTN, TY = kGBM / kGTM;
    __shared__ acc_t As[kGBK][kGBM + 1];   // A tile, transposed: As[k][m]
    __shared__ acc_t Bs[kGBK][kGBN];
    const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;

    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int lo = owner[tile];                        // the member owning this tile
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
            // all of a thread's loads of the step first, then the stores
            constexpr int P = kGBM * kGBK / kGThreads;    // = kGBK * kGBN / kGThreads
            acc_t va[P], vb[P];
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const int e = threadIdx.x + q * kGThreads;
                const int ra = e / kGBK, ca = e % kGBK, rb = e / kGBN, cb = e % kGBN;
                va[q] = (m0 + ra < M && k0 + ca < K) ? Num<T>::to_acc(A[(m0 + ra) * K + k0 + ca]) : acc_t(0);
                vb[q] = (k0 + rb < K && n0 + cb < N) ? Num<T>::to_acc(B[(k0 + rb) * N + n0 + cb]) : acc_t(0);
            }
            __syncthreads();   // the previous step (or tile) is done with the tiles
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const int e = threadIdx.x + q * kGThreads;
                As[e % kGBK][e / kGBK] = va[q];
                Bs[e / kGBN][e % kGBN] = vb[q];
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

// FLOAT16 / BFLOAT16 members: the same tiles on the tensor cores.  Four warps
// per 64 x 64 tile, each a 32 x 32 quarter from 2 x 4 mma.sync.m16n8k16
// products per 16-deep step (float32 accumulators).  The 64 x 32 A slice and
// 32 x 64 B slice of a step are staged as 16-bit values (zero outside the
// member), rows padded so that the ldmatrix row addresses of one 8 x 8
// matrix fall in eight different bank groups; A fragments by ldmatrix, B
// fragments by ldmatrix.trans from the row-major [k][n] slice.
constexpr int kMK = 32;                 // K per staged slice
constexpr int kALd = kMK + 8;           // A slice row: 40 halves (80 bytes)
constexpr int kBLd = kGBN + 8;          // B slice row: 72 halves (144 bytes)

__device__ __forceinline__ void g_ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void g_ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
template <bool BF16>
__device__ __forceinline__ void g_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if (BF16)
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

template <typename T>
__global__ void __launch_bounds__(128)
grouped_mma_kernel(const GDesc* __restrict__ desc, const int* __restrict__ owner, int64_t total_tiles,
                   const void* const* __restrict__ Aptr, const void* const* __restrict__ Bptr,
                   void* const* __restrict__ Yptr) {
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    __shared__ __align__(16) unsigned short As[kGBM][kALd];
    __shared__ __align__(16) unsigned short Bs[kMK][kBLd];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;    // this warp's quarter of the tile
    const uint32_t as_base = static_cast<uint32_t>(__cvta_generic_to_shared(&As[0][0]));
    const uint32_t bs_base = static_cast<uint32_t>(__cvta_generic_to_shared(&Bs[0][0]));

    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int lo = owner[tile];                        // the member owning this tile
        const GDesc d = desc[lo];
        const int64_t local = tile - d.tile_begin;
        const int64_t m0 = (local / d.tiles_n) * kGBM, n0 = (local % d.tiles_n) * kGBN;
        const int64_t M = d.m, N = d.n, K = d.k;
        const unsigned short* __restrict__ A = static_cast<const unsigned short*>(Aptr[lo]);
        const unsigned short* __restrict__ B = static_cast<const unsigned short*>(Bptr[lo]);
        T* __restrict__ Y = static_cast<T*>(Yptr[lo]);

        float acc[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
        for (int64_t k0 = 0; k0 < K; k0 += kMK) {
            // the slice's elements are all requested before any is stored, so
            // the loads of a thread overlap instead of queueing one by one
            constexpr int PA = kGBM * kMK / 128, PB = kMK * kGBN / 128;
            unsigned short va[PA], vb[PB];
#pragma unroll
            for (int q = 0; q < PA; ++q) {
                const int e = threadIdx.x + q * 128, r = e / kMK, c = e % kMK;
                const int64_t gm = m0 + r, gk = k0 + c;
                va[q] = (gm < M && gk < K) ? A[gm * K + gk] : (unsigned short)0;
            }
#pragma unroll
            for (int q = 0; q < PB; ++q) {
                const int e = threadIdx.x + q * 128, r = e / kGBN, c = e % kGBN;
                const int64_t gk = k0 + r, gn = n0 + c;
                vb[q] = (gk < K && gn < N) ? B[gk * N + gn] : (unsigned short)0;
            }
            __syncthreads();   // the previous slice (or tile) is no longer read
#pragma unroll
            for (int q = 0; q < PA; ++q) {
                const int e = threadIdx.x + q * 128;
                As[e / kMK][e % kMK] = va[q];
            }
#pragma unroll
            for (int q = 0; q < PB; ++q) {
                const int e = threadIdx.x + q * 128;
                Bs[e / kGBN][e % kGBN] = vb[q];
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < kMK; kk += 16) {
                uint32_t a[2][4], b[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    // matrices: rows 0-7 / 8-15 at k, then at k + 8
                    const int r = wm + 16 * i + (lane & 15), c = kk + (lane >> 4) * 8;
                    g_ldsm_x4(as_base + (uint32_t)((r * kALd + c) * 2), a[i]);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // matrices: k 0-7 / 8-15 of columns n, then of columns n + 8
                    const int r = kk + (lane & 15), c = wn + 16 * j + (lane >> 4) * 8;
                    g_ldsm_x4_t(bs_base + (uint32_t)((r * kBLd + c) * 2), b[j]);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        g_mma<BF16>(acc[i][j], a[i], b[j >> 1][2 * (j & 1)], b[j >> 1][2 * (j & 1) + 1]);
            }
        }
        // fragment (g, t): rows g and g + 8 of each 16-row block, columns 2t, 2t + 1
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t gm = m0 + wm + 16 * i + g + 8 * h;
                    const int64_t gn = n0 + wn + 8 * j + 2 * t;
                    if (gm >= M) continue;
                    if (gn < N) Y[gm * N + gn] = Num<T>::from_acc(acc[i][j][2 * h]);
                    if (gn + 1 < N) Y[gm * N + gn + 1] = Num<T>::from_acc(acc[i][j][2 * h + 1]);
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
    int device;                  // -1 until the tables are on a device
    olc::GDesc* desc_dev;
    int* owner_dev;              // member of every tile
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
    // the descriptor table and, for every tile, the member that owns it
    std::vector<int> owner;
    try {
        owner.resize((size_t)p->total_tiles);
    } catch (const std::bad_alloc&) {
        return OLC_ERR_OOM;
    }
    for (int i = 0; i < p->count; ++i) {
        const int64_t end = i + 1 < p->count ? p->desc[i + 1].tile_begin : p->total_tiles;
        for (int64_t t = p->desc[i].tile_begin; t < end; ++t) owner[(size_t)t] = i;
    }
    void* mem = nullptr;
    const size_t bytes = sizeof(olc::GDesc) * (size_t)p->count;
    const size_t obytes = sizeof(int) * owner.size();
    cudaError_t e = cudaMalloc(&mem, bytes + obytes);
    if (e == cudaSuccess) e = cudaMemcpy(mem, p->desc.data(), bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && obytes)
        e = cudaMemcpy(static_cast<unsigned char*>(mem) + bytes, owner.data(), obytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (mem) cudaFree(mem);
        return grouped_from_cuda(e);
    }
    p->owner_dev = reinterpret_cast<int*>(static_cast<unsigned char*>(mem) + bytes);
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
    // every member's A, B and Y within 2^62 bytes (element offsets stay in
    // int64), and all members' tiles numbered in an int owner table
    const int64_t eb = (dtype == OLC_DOUBLE) ? 8 : (dtype == OLC_FLOAT) ? 4 : 2;
    int64_t t = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t pairs[3][2] = {{m[i], k[i]}, {k[i], n[i]}, {m[i], n[i]}};
        for (const auto& d : pairs) {
            int64_t bytes = 0;
            if (d[0] != 0 && d[1] != 0 &&
                (__builtin_mul_overflow(d[0], d[1], &bytes) || __builtin_mul_overflow(bytes, eb, &bytes) ||
                 bytes > (int64_t(1) << 62)))
                return OLC_ERR_INVALID;
        }
        t += olc::ceil_div(m[i], olc::kGBM) * olc::ceil_div(n[i], olc::kGBN);
        if (t > 0x7fffffffLL) return OLC_ERR_INVALID;
    }
    olc_grouped_plan* p = new (std::nothrow) olc_grouped_plan;
    if (!p) return OLC_ERR_OOM;
    p->dtype = dtype;
    p->count = count;
    p->device = -1;
    p->desc_dev = nullptr;
    p->owner_dev = nullptr;
    p->sm_count = 0;
    try {
        p->desc.resize((size_t)count);
    } catch (const std::bad_alloc&) {
        delete p;
        return OLC_ERR_OOM;
    }
    t = 0;
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
    cudaError_t e;
    if (plan->dtype == OLC_FLOAT16 || plan->dtype == OLC_BFLOAT16) {
        const int64_t grid = olc::min64(plan->total_tiles, (int64_t)plan->sm_count * 8);
        if (plan->dtype == OLC_FLOAT16)
            olc::grouped_mma_kernel<__half><<<(unsigned)grid, 128, 0, s>>>(p->desc_dev, p->owner_dev,
                                                                          p->total_tiles, A, B, Y);
        else
            olc::grouped_mma_kernel<__nv_bfloat16><<<(unsigned)grid, 128, 0, s>>>(
                p->desc_dev, p->owner_dev, p->total_tiles, A, B, Y);
        e = cudaGetLastError();
    } else {
        const int64_t grid = olc::min64(plan->total_tiles, (int64_t)plan->sm_count * 4);
        e = olc::dispatch_dtype(plan->dtype, [&](auto tag) {
            using T = decltype(tag);
            olc::grouped_kernel<T><<<(unsigned)grid, olc::kGThreads, 0, s>>>(
                p->desc_dev, p->owner_dev, p->total_tiles, A, B, Y);
            return cudaGetLastError();
        });
    }
    return grouped_from_cuda(e);
}

}  // extern "C"
