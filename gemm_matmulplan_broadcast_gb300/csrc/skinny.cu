// Skinny kernels: SKINNY_M (few output rows) and SKINNY_N (few output
// columns), plus the GENERAL_SIMT launcher that routes by vectorisability.
//
// "Gemm and MatMul Performance Roadmap", section "Target computation
// algorithm", the algorithm-by-shape table: for M == 1 or very small M a
// GEMV/skinny-M kernel that streams B once and vectorises across N; for
// N == 1 or very small N a dot/GEMV kernel that vectorises the K reduction.
// Both are bound by HBM bandwidth (arithmetic intensity of a few flop/byte),
// so the kernels are built around wide coalesced loads and enough loads in
// flight, not around arithmetic.
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace olc {

cudaError_t launch_general_simt_generic(olc_dtype dt, const Problem& p, cudaStream_t stream);
cudaError_t launch_general_simt_fast(olc_dtype dt, const Problem& p, cudaStream_t stream, int splits,
                                     const Workspace* ws);
bool general_simt_fast_ok(olc_dtype dt, int64_t N, int64_t K);

bool general_simt_vectorizable(olc_dtype dt, int64_t N, int64_t K) {
    return general_simt_fast_ok(dt, N, K);
}

cudaError_t launch_general_simt(olc_dtype dt, const Problem& p, cudaStream_t stream, int splits,
                                const Workspace* ws) {
    if (general_simt_fast_ok(dt, p.N, p.K)) return launch_general_simt_fast(dt, p, stream, splits, ws);
    return launch_general_simt_generic(dt, p, stream);
}

// ===========================================================================
// SKINNY_M
//
// Block = KW warps.  Lane l of every warp owns VEC consecutive output columns
// (one 16-byte vector of each B row; 8 or 4 bytes for one-byte elements with
// 4 or more rows); the block covers 32 * VEC columns.  The KW warps split the
// block's K range; within its range a warp walks k in ascending order,
// loading B[k][cols] as one vector per lane and the MR rows' next 8 values
// of A (the same addresses for all lanes, so broadcast loads, kept packed and
// widened two k positions at a time), and keeps an MR x VEC accumulator tile
// in registers (float accumulators as packed pairs for fma.rn.f32x2).  The warps' tiles are
// summed in shared memory in warp order.  With ksplit > 1 the grid also
// splits K across blocks: each block writes its partial tile to the
// workspace, and the last block to arrive for a column group (counted with an
// atomic) adds the partials in split order 0..ksplit-1 -- the same order
// whichever block arrives last, so results are reproducible run to run.

constexpr int kSkinnyMMax = 16;

int skinny_m_max_rows() { return kSkinnyMMax; }

// Columns per lane: one 16-byte B vector, except for one-byte elements with
// four or more rows, where 16 columns per lane would hold 16 * MR float
// accumulators: 8 columns (8-byte loads) for 4 rows, 4 columns (4-byte
// loads) from 8 rows on.
template <typename T, int MR>
struct SkinnyMVec {
    static constexpr int N = sizeof(T) != 1 ? 16 / (int)sizeof(T) : (MR <= 2 ? 16 : MR == 4 ? 8 : 4);
    static constexpr int WORDS = N * (int)sizeof(T) / 4;   // 32-bit words per lane per B row
};

// WORDS consecutive 32-bit words through the read-only path, in one load
template <int WORDS>
__device__ __forceinline__ void ldg_words(const void* ptr, uint32_t (&w)[WORDS]) {
    if constexpr (WORDS == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(ptr));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (WORDS == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(ptr));
        w[0] = v.x; w[1] = v.y;
    } else {
        static_assert(WORDS == 1, "1, 2 or 4 words");
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(ptr));
    }
}

// One output row's VEC accumulators of a lane.  Float accumulators are kept
// as packed column pairs and updated with fma.rn.f32x2 (two round-to-nearest
// FMAs per issue slot, per element the same arithmetic as fmaf); double
// accumulators use DFMA.
template <typename A, int VEC>
struct AccRow {
    A v[VEC];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int c = 0; c < VEC; ++c) v[c] = A(0);
    }
    __device__ __forceinline__ void fma_row(A a, const A (&b)[VEC]) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) v[c] = fma(a, b[c], v[c]);
    }
    __device__ __forceinline__ A get(int c) const { return v[c]; }
};
template <int VEC>
struct AccRow<float, VEC> {
    static_assert(VEC % 2 == 0, "column pairs");
    unsigned long long v[VEC / 2];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int c = 0; c < VEC / 2; ++c) v[c] = 0ull;
    }
    __device__ __forceinline__ void fma_row(float a, const unsigned long long (&b2)[VEC / 2]) {
        const unsigned long long a2 = pack_f2(a, a);
#pragma unroll
        for (int c = 0; c < VEC / 2; ++c) fma_f2(v[c], a2, b2[c]);
    }
    __device__ __forceinline__ float get(int c) const {
        float lo, hi;
        unpack_f2(v[c / 2], lo, hi);
        return (c & 1) ? hi : lo;
    }
};

// B operand row as the accumulator row consumes it: packed pairs for float
template <typename A, int VEC>
struct BRow {
    A b[VEC];
    __device__ __forceinline__ void set(const A (&x)[VEC]) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) b[c] = x[c];
    }
    __device__ __forceinline__ const A (&operand() const)[VEC] { return b; }
};
template <int VEC>
struct BRow<float, VEC> {
    unsigned long long b2[VEC / 2];
    __device__ __forceinline__ void set(const float (&x)[VEC]) {
#pragma unroll
        for (int c = 0; c < VEC / 2; ++c) b2[c] = pack_f2(x[2 * c], x[2 * c + 1]);
    }
    __device__ __forceinline__ const unsigned long long (&operand() const)[VEC / 2] { return b2; }
};

// Bits of one element and back, for A rows kept as raw 32-bit words
// (elements packed little-endian, 8-byte elements over two words).
template <typename T>
struct ElemBits;
template <>
struct ElemBits<float> {
    static __device__ __forceinline__ uint32_t bits(float v) { return __float_as_uint(v); }
};
template <>
struct ElemBits<__half> {
    static __device__ __forceinline__ uint32_t bits(__half v) { return __half_as_ushort(v); }
};
template <>
struct ElemBits<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t bits(__nv_bfloat16 v) { return __bfloat16_as_ushort(v); }
};
template <int FMT>
struct ElemBits<F8<FMT>> {
    static __device__ __forceinline__ uint32_t bits(F8<FMT> v) { return v.bits; }
};

// element u of a raw row, stored into the words
template <typename T, int AW>
__device__ __forceinline__ void put_elem(uint32_t (&w)[AW], int u, T v) {
    if constexpr (sizeof(T) == 8) {
        const unsigned long long b = (unsigned long long)__double_as_longlong(v);
        w[2 * u] = (uint32_t)b;
        w[2 * u + 1] = (uint32_t)(b >> 32);
    } else {
        constexpr int PER = 4 / (int)sizeof(T);
        const uint32_t b = ElemBits<T>::bits(v) << (8 * (int)sizeof(T) * (u % PER));
        w[u / PER] = (u % PER == 0) ? b : (w[u / PER] | b);
    }
}

// elements u0 and u0 + 1 (UP = 2: one- and two-byte types) or u0 alone
// (UP = 1) of a raw row, in the accumulator type
template <typename T, int AW, int UP>
__device__ __forceinline__ void get_elems(const uint32_t (&w)[AW], int u0,
                                          typename Num<T>::acc_t (&out)[UP]) {
    if constexpr (sizeof(T) == 8) {
        out[0] = __hiloint2double((int)w[2 * u0 + 1], (int)w[2 * u0]);
    } else if constexpr (sizeof(T) == 4) {
        out[0] = __uint_as_float(w[u0]);
    } else if constexpr (sizeof(T) == 2) {
        const uint32_t x = w[u0 / 2];
        if constexpr (std::is_same<T, __half>::value) {
            out[0] = __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
            out[1] = __half2float(__ushort_as_half((unsigned short)(x >> 16)));
        } else {
            out[0] = __bfloat162float(__ushort_as_bfloat16((unsigned short)(x & 0xFFFFu)));
            out[1] = __bfloat162float(__ushort_as_bfloat16((unsigned short)(x >> 16)));
        }
    } else {
        const uint32_t x = (w[u0 / 4] >> (8 * (u0 % 4))) & 0xFFFFu;
        const uint32_t pair[1] = {x};
        float four[4];
        fp8_decode_words<T::kFormat, 1>(pair, four);   // bytes 2 and 3 are zero
        out[0] = four[0];
        out[1] = four[1];
    }
}

// the accumulator-type values of the elements packed in `w`
template <typename T, int WORDS>
__device__ __forceinline__ void widen_words(const uint32_t (&w)[WORDS],
                                            typename Num<T>::acc_t (&out)[WORDS * 4 / sizeof(T)]) {
    if constexpr (sizeof(T) == 1) {
        fp8_decode_words<T::kFormat, WORDS>(w, out);
    } else {
        const T* e = reinterpret_cast<const T*>(w);
#pragma unroll
        for (int v = 0; v < (int)(WORDS * 4 / sizeof(T)); ++v) out[v] = Num<T>::to_acc(e[v]);
    }
}

// warps splitting K in a block; one-byte operands, whose lanes hold fewer
// columns from 4 rows on, keep more warps (and more loads in flight)
template <typename T, int MR>
struct SkinnyMConfig {
    static constexpr int KW = sizeof(T) == 1 ? (MR <= 8 ? 8 : 4) : (MR <= 4 ? 8 : (MR <= 8 ? 4 : 2));
};

// End of a skinny-M block: sum the KW warps' MR x COLS tiles (red) in warp
// order; with ksplit == 1 store them through the epilogue, otherwise file the
// block's partial tile in the workspace and let the last block of the column
// group to arrive (an atomic count) add the partials in split order
// 0..ksplit-1 -- the same order whichever block arrives last, so results are
// reproducible run to run.  Every thread of the block calls it.
template <typename T, int MR, int COLS, int KW>
__device__ __forceinline__ void skinny_m_finish(const Problem& p,
                                                const typename Num<T>::acc_t (&red)[KW][MR][COLS],
                                                unsigned int& am_last, int64_t item, int64_t cg, int split,
                                                int ksplit, int64_t col_groups, const Workspace& ws,
                                                typename Num<T>::out_t* __restrict__ Y) {
    using acc_t = typename Num<T>::acc_t;
    using out_t = typename Num<T>::out_t;
    const int64_t M = p.M, N = p.N;
    // thread t owns entries t, t + NT, ...
    constexpr int NT = KW * 32;
    constexpr int ENTRIES = MR * COLS;
    constexpr int Q = (ENTRIES + NT - 1) / NT;
    acc_t part[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = threadIdx.x + q * NT;
        acc_t s = acc_t(0);
        if (e < ENTRIES) {
            const int i = e / COLS, c = e % COLS;
            s = red[0][i][c];
#pragma unroll
            for (int w = 1; w < KW; ++w) s += red[w][i][c];
        }
        part[q] = s;
    }

    if (ksplit == 1) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int e = threadIdx.x + q * NT;
            if (e >= ENTRIES) continue;
            const int i = e / COLS, c = e % COLS;
            const int64_t col = cg * COLS + c;
            if (i < M && col < N)
                Y[i * N + col] = Num<T>::from_acc(apply_epilogue<out_t>(p.epi, part[q], i, col, Y + i * N + col));
        }
        return;
    }

    // cross-block split: partial tile -> workspace, last arrival reduces
    acc_t* P = static_cast<acc_t*>(ws.partials);
    const int64_t tile = item * col_groups + cg;
    acc_t* mine = P + (tile * ksplit + split) * ENTRIES;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = threadIdx.x + q * NT;
        if (e < ENTRIES) mine[e] = part[q];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(ws.counters + tile, 1u);
        am_last = (prev == (unsigned int)ksplit - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!am_last) return;
    __threadfence();
    const acc_t* all = P + tile * ksplit * ENTRIES;
    for (int e = threadIdx.x; e < ENTRIES; e += NT) {
        acc_t s = __ldcg(all + e);
        for (int t = 1; t < ksplit; ++t) s += __ldcg(all + (int64_t)t * ENTRIES + e);
        const int i = e / COLS, c = e % COLS;
        const int64_t col = cg * COLS + c;
        if (i < M && col < N)
            Y[i * N + col] = Num<T>::from_acc(apply_epilogue<out_t>(p.epi, s, i, col, Y + i * N + col));
    }
    if (threadIdx.x == 0) ws.counters[tile] = 0u;   // ready for the next launch
}

template <typename T, int MR>
__global__ void __launch_bounds__(SkinnyMConfig<T, MR>::KW * 32)
skinny_m_kernel(Problem p, int64_t col_groups, int ksplit, int64_t kslice, Workspace ws,
                int a_vec_ok) {
    using acc_t = typename Num<T>::acc_t;
    using out_t = typename Num<T>::out_t;    // float32 for 8-bit float operands
    constexpr int VEC = SkinnyMVec<T, MR>::N;
    constexpr int WORDS = SkinnyMVec<T, MR>::WORDS;
    constexpr int KW = SkinnyMConfig<T, MR>::KW;
    constexpr int COLS = 32 * VEC;
    constexpr int KU = 8;                    // k rows per step: 8 B vectors in flight per lane
    constexpr int AW = KU * (int)sizeof(T) / 4;           // 32-bit words of A per row per step
    constexpr int UP = sizeof(T) <= 2 ? 2 : 1;             // k rows decoded together from A
    __shared__ acc_t red[KW][MR][COLS];
    __shared__ unsigned int am_last;

    const int64_t per_item = col_groups * ksplit;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int split = (int)(rem / col_groups);
    const int64_t cg = rem % col_groups;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    out_t* __restrict__ Y = static_cast<out_t*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t col0 = cg * COLS + (int64_t)lane * VEC;
    const bool col_ok = col0 < N;   // N is a multiple of VEC
    // this block's K range (kslice is a multiple of KU), then this warp's
    // share of it, also a multiple of KU
    const int64_t kb0 = (int64_t)split * kslice;
    const int64_t kb1 = min64(K, kb0 + kslice);
    const int64_t wlen = ceil_div(ceil_div(max64(kb1 - kb0, 0), KW), KU) * KU;
    const int64_t k0 = min64(kb1, kb0 + warp * wlen);
    const int64_t k1 = min64(kb1, k0 + wlen);

    AccRow<acc_t, VEC> acc[MR];
#pragma unroll
    for (int i = 0; i < MR; ++i) acc[i].zero();

    if (col_ok) {
        const T* bp = B + col0;
        int64_t k = k0;
        for (; k + KU <= k1; k += KU) {
            uint32_t bw[KU][WORDS];
#pragma unroll
            for (int u = 0; u < KU; ++u) ldg_words<WORDS>(bp + (k + u) * N, bw[u]);
            // A rows kept as raw words, decoded a k pair at a time: MR x KU
            // decoded values would take most of the registers at 8-16 rows
            uint32_t araw[MR][AW];
#pragma unroll
            for (int i = 0; i < MR; ++i) {
                if (i < M) {
                    if (a_vec_ok) {
                        if constexpr (AW == 2) {
                            const uint2 av = __ldg(reinterpret_cast<const uint2*>(A + i * K + k));
                            araw[i][0] = av.x;
                            araw[i][1] = av.y;
                        } else {
#pragma unroll
                            for (int q = 0; q < AW / 4; ++q) {
                                const uint4 av = __ldg(reinterpret_cast<const uint4*>(A + i * K + k) + q);
                                araw[i][4 * q] = av.x;
                                araw[i][4 * q + 1] = av.y;
                                araw[i][4 * q + 2] = av.z;
                                araw[i][4 * q + 3] = av.w;
                            }
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < KU; ++u) put_elem<T, AW>(araw[i], u, ldg_elem(A + i * K + k + u));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < AW; ++q) araw[i][q] = 0u;
                }
            }
#pragma unroll
            for (int u0 = 0; u0 < KU; u0 += UP) {
                acc_t a[MR][UP];
#pragma unroll
                for (int i = 0; i < MR; ++i) get_elems<T, AW, UP>(araw[i], u0, a[i]);
#pragma unroll
                for (int uu = 0; uu < UP; ++uu) {
                    acc_t b[VEC];
                    widen_words<T, WORDS>(bw[u0 + uu], b);
                    BRow<acc_t, VEC> br;
                    br.set(b);
#pragma unroll
                    for (int i = 0; i < MR; ++i) acc[i].fma_row(a[i][uu], br.operand());
                }
            }
        }
        for (; k < k1; ++k) {
            uint32_t bw[WORDS];
            ldg_words<WORDS>(bp + k * N, bw);
            acc_t b[VEC];
            widen_words<T, WORDS>(bw, b);
            BRow<acc_t, VEC> br;
            br.set(b);
#pragma unroll
            for (int i = 0; i < MR; ++i)
                acc[i].fma_row(i < M ? Num<T>::to_acc(ldg_elem(A + i * K + k)) : acc_t(0), br.operand());
        }
    }
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) red[warp][i][lane * VEC + v] = acc[i].get(v);
    __syncthreads();

    skinny_m_finish<T, MR, COLS, KW>(p, red, am_last, item, cg, split, ksplit, col_groups, ws, Y);
}

// ===========================================================================
// SKINNY_M for E4M3FN / E5M2 operands on the warp-level MMA
//
// mma.sync.aligned.m16n8k32.row.col.f32.{e4m3,e5m2}: D[16 x 8] += A[16 x 32]
// * B[32 x 8] with float32 accumulation.  The MMA's 16 rows are the
// product's rows of A (at most 16, the rest zeros); its 32 K positions a
// 32-row chunk of B.  Lane (g, t) = (lane / 4, lane % 4) loads 8 bytes --
// columns 8 g .. 8 g + 7 of the warp's 64-column group -- from the chunk's B
// rows 4 t .. 4 t + 3 and 16 + 4 t .. 16 + 4 t + 3, the K positions its B
// fragment registers hold, and transposes each 4 x 4 byte block with byte
// permutes: register p of the result holds column 8 g + p at those four K
// positions, i.e. the B fragment of MMA p (p = 0..7), whose column n stands
// for product column 8 n + p.  The eight MMAs of a chunk cover the 64
// columns and share one A fragment (rows g and g + 8 at the lane's K
// positions, one 4-byte load each).  So B is read once, in the layout it is
// stored in.  Each lane keeps F8_RING chunks of loads (B and A) in a
// register ring, issuing chunk c + F8_RING - 1 before the MMAs of chunk c:
// at HBM rates a load takes microseconds to return, and the bytes in flight
// per SM set the bandwidth.  Blocks of kF8MmaWarps warps split K as the SIMT
// kernel's do and end the same way (skinny_m_finish), or, as the split-K of
// small outputs (MT = 2 tiles for up to 32 rows, about one K slice per SM),
// with two reduction levels (skinny_m_finish_grouped).

constexpr int kF8MmaWarps = 4;
constexpr int kF8MmaCols = 64;
constexpr int F8_RING = 4;

template <int FMT>
__device__ __forceinline__ void mma_f8_m16n8k32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1) {
    if constexpr (FMT == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        static_assert(FMT == 1, "E4M3FN or E5M2");
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e5m2.e5m2.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// 4 x 4 byte transpose: out[q] = byte q of r0, r1, r2, r3 (in that order)
__device__ __forceinline__ void transpose4x4_bytes(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                                   uint32_t (&out)[4]) {
    const uint32_t x = __byte_perm(r0, r1, 0x5140), y = __byte_perm(r2, r3, 0x5140);
    const uint32_t x2 = __byte_perm(r0, r1, 0x7362), y2 = __byte_perm(r2, r3, 0x7362);
    out[0] = __byte_perm(x, y, 0x5410);
    out[1] = __byte_perm(x, y, 0x7632);
    out[2] = __byte_perm(x2, y2, 0x5410);
    out[3] = __byte_perm(x2, y2, 0x7632);
}

// one chunk's operands in a lane: 8 B rows of 8 bytes, the A fragments of
// MT 16-row tiles
template <int MT>
struct F8Chunk {
    uint2 b[8];
    uint32_t a[MT][4];
};

// acc[q] = sum over slices t = 0..n-1 (ascending) of src[t * stride + q * NT]
// for this thread's entries (ok[q]; others give 0); the loads of UNR slices
// are issued together, so a sum over many slices costs n / UNR round trips
// to L2 instead of n.
template <int Q, int NT, int UNR = 4>
__device__ __forceinline__ void sum_slices(float (&acc)[Q], const float* __restrict__ src, int n, int64_t stride,
                                           const bool (&ok)[Q]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) acc[q] = ok[q] ? __ldcg(src + q * NT) : 0.0f;
    int t = 1;
    for (; t + UNR <= n; t += UNR) {
        float x[UNR][Q];
#pragma unroll
        for (int u = 0; u < UNR; ++u)
#pragma unroll
            for (int q = 0; q < Q; ++q) x[u][q] = ok[q] ? __ldcg(src + (int64_t)(t + u) * stride + q * NT) : 0.0f;
#pragma unroll
        for (int u = 0; u < UNR; ++u)
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[q] += x[u][q];
    }
    for (; t < n; ++t)
#pragma unroll
        for (int q = 0; q < Q; ++q) acc[q] += ok[q] ? __ldcg(src + (int64_t)t * stride + q * NT) : 0.0f;
}

// Two-level end of a split over K (sgroup > 0): each block files its partial
// tile; the last block of each group of sgroup consecutive slices (an atomic
// count) adds the group's partials in slice order into a group sum; the last
// group to finish adds the group sums in group order and stores through the
// epilogue.  Fixed orders at both levels, so results are reproducible run to
// run; one level would leave a single block reading every slice's partial.
// Workspace: partials [tiles][ksplit][ENTRIES], then group sums
// [tiles][groups][ENTRIES]; counters [tiles][groups + 1], zero between
// launches (the last arrivals reset them).  Only columns below N are filed
// and summed.
template <typename T, int MR, int COLS, int KW>
__device__ __forceinline__ void skinny_m_finish_grouped(const Problem& p, const float (&red)[KW][MR][COLS],
                                                        unsigned int& am_last, int64_t item, int64_t cg,
                                                        int split, int ksplit, int sgroup, int64_t col_groups,
                                                        const Workspace& ws, float* __restrict__ Y) {
    constexpr int NT = KW * 32;
    constexpr int ENTRIES = MR * COLS;
    static_assert(ENTRIES % NT == 0, "whole entries per thread");
    constexpr int Q = ENTRIES / NT;
    const int64_t M = p.M, N = p.N;
    const int ncols = (int)min64(COLS, N - cg * COLS);
    const int64_t tile = item * col_groups + cg;
    const int64_t tiles = col_groups * p.items;
    const int groups = (ksplit + sgroup - 1) / sgroup;
    float* P = static_cast<float*>(ws.partials);
    float* G = P + tiles * ksplit * ENTRIES;
    unsigned int* cnt = ws.counters + tile * (groups + 1);

    bool ok[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) ok[q] = (threadIdx.x + q * NT) % COLS < ncols;
    float* mine = P + (tile * ksplit + split) * ENTRIES;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = threadIdx.x + q * NT;
        if (!ok[q]) continue;
        const int i = e / COLS, c = e % COLS;
        float v = red[0][i][c];
#pragma unroll
        for (int w = 1; w < KW; ++w) v += red[w][i][c];
        mine[e] = v;
    }
    __threadfence();
    __syncthreads();
    const int grp = split / sgroup;
    const int s0 = grp * sgroup, sn = min(sgroup, ksplit - s0);
    if (threadIdx.x == 0) am_last = (atomicAdd(cnt + grp, 1u) == (unsigned int)sn - 1) ? 1u : 0u;
    __syncthreads();
    if (!am_last) return;
    __threadfence();
    float acc[Q];
    sum_slices<Q, NT>(acc, P + (tile * ksplit + s0) * ENTRIES + threadIdx.x, sn, ENTRIES, ok);
    float* gsum = G + (tile * groups + grp) * ENTRIES;
#pragma unroll
    for (int q = 0; q < Q; ++q)
        if (ok[q]) gsum[threadIdx.x + q * NT] = acc[q];
    if (threadIdx.x == 0) cnt[grp] = 0u;   // ready for the next launch
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) am_last = (atomicAdd(cnt + groups, 1u) == (unsigned int)groups - 1) ? 1u : 0u;
    __syncthreads();
    if (!am_last) return;
    __threadfence();
#pragma unroll
    for (int q = 0; q < Q; ++q) ok[q] = ok[q] && (threadIdx.x + q * NT) / COLS < M;
    sum_slices<Q, NT>(acc, G + tile * groups * ENTRIES + threadIdx.x, groups, ENTRIES, ok);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        if (!ok[q]) continue;
        const int e = threadIdx.x + q * NT;
        const int i = e / COLS;
        const int64_t col = cg * COLS + e % COLS;
        Y[i * N + col] = apply_epilogue<float>(p.epi, acc[q], i, col, Y + i * N + col);
    }
    if (threadIdx.x == 0) cnt[groups] = 0u;
}

template <int FMT, int MT>
__global__ void __launch_bounds__(kF8MmaWarps * 32, MT == 1 ? 3 : 2)
skinny_m_f8_mma_kernel(Problem p, int64_t col_groups, int ksplit, int64_t kslice, int sgroup, Workspace ws,
                       int a_vec_ok) {
    using T = F8<FMT>;
    constexpr int KW = kF8MmaWarps;
    constexpr int COLS = kF8MmaCols;
    constexpr int MR = 16 * MT;
    constexpr int R = F8_RING;
    __shared__ float red[KW][MR][COLS];
    __shared__ unsigned int am_last;

    const int64_t per_item = col_groups * ksplit;
    const int64_t item = blockIdx.x / per_item;
    const int64_t rem = blockIdx.x % per_item;
    const int split = (int)(rem / col_groups);
    const int64_t cg = rem % col_groups;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const unsigned char* __restrict__ A = static_cast<const unsigned char*>(p.A) + a_off;
    const unsigned char* __restrict__ B = static_cast<const unsigned char*>(p.B) + b_off;
    float* __restrict__ Y = static_cast<float*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t col0 = cg * COLS + 8 * g;    // this lane's 8 columns
    const bool col_ok = col0 < N;             // N is a multiple of 16
    // this block's K range (kslice is a multiple of 32), then this warp's
    // share of it, also a multiple of 32
    const int64_t kb0 = (int64_t)split * kslice;
    const int64_t kb1 = min64(K, kb0 + kslice);
    const int64_t wlen = ceil_div(ceil_div(max64(kb1 - kb0, 0), KW), 32) * 32;
    const int64_t k0 = min64(kb1, kb0 + warp * wlen);
    const int64_t k1 = min64(kb1, k0 + wlen);

    // A[row][kk .. kk + 3] packed little-endian; zero past k1 and past M
    auto a_word = [&](int row, int64_t kk) -> uint32_t {
        if (row >= M) return 0u;
        const unsigned char* ar = A + row * K;
        if (a_vec_ok && kk + 4 <= k1) return __ldg(reinterpret_cast<const unsigned int*>(ar + kk));
        uint32_t w = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (kk + i < k1) w |= (uint32_t)__ldg(ar + kk + i) << (8 * i);
        return w;
    };
    // B rows kc + 4t + j (j < 4) and kc + 16 + 4t + j of the lane's columns,
    // and the A fragment; rows at or past k1 (another warp's range, or past
    // K) read as zeros
    const unsigned char* __restrict__ Bl = B + (int64_t)(4 * t) * N + col0;   // row 4t, lane's columns
    auto load_chunk = [&](int64_t kc, F8Chunk<MT>& c) {
        const unsigned char* bk = Bl + kc * N;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int dr = j < 4 ? j : 16 + (j - 4);
            const int64_t r = kc + 4 * t + dr;
            c.b[j] = (col_ok && r < k1) ? __ldg(reinterpret_cast<const uint2*>(bk + (int64_t)dr * N))
                                        : make_uint2(0u, 0u);
        }
        if (kc < k1) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                c.a[mt][0] = a_word(16 * mt + g, kc + 4 * t);
                c.a[mt][1] = a_word(16 * mt + g + 8, kc + 4 * t);
                c.a[mt][2] = a_word(16 * mt + g, kc + 16 + 4 * t);
                c.a[mt][3] = a_word(16 * mt + g + 8, kc + 16 + 4 * t);
            }
        }
    };

    float d[MT][8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) d[mt][q][i] = 0.0f;

    F8Chunk<MT> ring[R];
#pragma unroll
    for (int r = 0; r < R - 1; ++r) load_chunk(k0 + 32 * r, ring[r]);
    for (int64_t kc = k0; kc < k1; kc += 32 * R) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t kcur = kc + 32 * r;
            load_chunk(kcur + 32 * (R - 1), ring[(r + R - 1) % R]);
            if (kcur < k1) {
                const F8Chunk<MT>& c = ring[r];
                // lo: K positions 4t..4t+3, hi: 16+4t..; [0]: columns 0-3, [1]: 4-7
                uint32_t lo[2][4], hi[2][4];
                transpose4x4_bytes(c.b[0].x, c.b[1].x, c.b[2].x, c.b[3].x, lo[0]);
                transpose4x4_bytes(c.b[0].y, c.b[1].y, c.b[2].y, c.b[3].y, lo[1]);
                transpose4x4_bytes(c.b[4].x, c.b[5].x, c.b[6].x, c.b[7].x, hi[0]);
                transpose4x4_bytes(c.b[4].y, c.b[5].y, c.b[6].y, c.b[7].y, hi[1]);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mma_f8_m16n8k32<FMT>(d[mt][q], c.a[mt], lo[q / 4][q % 4], hi[q / 4][q % 4]);
            }
        }
    }

    // MMA q's accumulator of tile mt: rows 16 mt + g and 16 mt + g + 8, MMA
    // columns 2t and 2t + 1, i.e. columns 8 (2t) + q and 8 (2t + 1) + q of
    // the group
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            red[warp][16 * mt + g][16 * t + q] = d[mt][q][0];
            red[warp][16 * mt + g][16 * t + 8 + q] = d[mt][q][1];
            red[warp][16 * mt + g + 8][16 * t + q] = d[mt][q][2];
            red[warp][16 * mt + g + 8][16 * t + 8 + q] = d[mt][q][3];
        }
    __syncthreads();
    if (sgroup > 0 && ksplit > 1)
        skinny_m_finish_grouped<T, MR, COLS, KW>(p, red, am_last, item, cg, split, ksplit, sgroup, col_groups, ws,
                                                 Y);
    else
        skinny_m_finish<T, MR, COLS, KW>(p, red, am_last, item, cg, split, ksplit, col_groups, ws, Y);
}

static int round_rows(int64_t m) {
    return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16;
}

// bytes of one operand element (8-bit float types: 1)
static int64_t operand_bytes(olc_dtype dt) {
    return dt == OLC_DOUBLE ? 8 : dt == OLC_FLOAT ? 4 : (dt == OLC_FLOAT16 || dt == OLC_BFLOAT16) ? 2 : 1;
}

// columns per lane of the SIMT skinny-M kernel (SkinnyMVec on the device)
static int64_t skinny_m_vec(olc_dtype dt, int64_t M) {
    const int64_t eb = operand_bytes(dt);
    const int mr = round_rows(M);
    return eb != 1 ? 16 / eb : (mr <= 2 ? 16 : mr == 4 ? 8 : 4);
}

static int64_t skinny_m_col_groups(olc_dtype dt, int64_t M, int64_t N) {
    return ceil_div(N, 32 * skinny_m_vec(dt, M));
}

// the SIMT skinny-M kernel's element types: the four MatMul types and the
// 8-bit float formats (F8<FMT>, float32 output); `other` for any other type
template <typename R, typename F>
static R dispatch_skinny_m(olc_dtype dt, R other, F&& f) {
    switch (dt) {
        case OLC_FLOAT: return f(float{});
        case OLC_DOUBLE: return f(double{});
        case OLC_FLOAT16: return f(__half{});
        case OLC_BFLOAT16: return f(__nv_bfloat16{});
        case OLC_FLOAT8E4M3FN: return f(F8<0>{});
        case OLC_FLOAT8E5M2: return f(F8<1>{});
        case OLC_FLOAT8E4M3FNUZ: return f(F8<2>{});
        case OLC_FLOAT8E5M2FNUZ: return f(F8<3>{});
    }
    return other;
}

template <typename T, int MR>
static int skinny_m_occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, skinny_m_kernel<T, MR>,
                                                      SkinnyMConfig<T, MR>::KW * 32, 0) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    return n > 0 ? n : 4;   // no device visible: assume four resident blocks
}

static int skinny_m_blocks_per_sm(olc_dtype dt, int64_t M) {
    const int mr = round_rows(M);
    return dispatch_skinny_m(dt, 4, [&](auto tag) -> int {
        using T = decltype(tag);
        switch (mr) {
            case 1: return skinny_m_occupancy<T, 1>();
            case 2: return skinny_m_occupancy<T, 2>();
            case 4: return skinny_m_occupancy<T, 4>();
            case 8: return skinny_m_occupancy<T, 8>();
            default: return skinny_m_occupancy<T, 16>();
        }
    });
}

// Number of K slices across blocks.  The grid is groups * splits blocks and
// runs in waves of sm_count * (resident blocks per SM); a last wave that is
// mostly empty costs as much as a full one, so pick the split with the best
// wave fill, discounted by the extra partial-tile traffic it causes.
// FLOAT16 / BFLOAT16 with 16-byte row strides: the tensor-core kernel with
// swapped operands streams B through its TMA ring; the rest: the SIMT kernel.
// FLOAT16 / BFLOAT16: the tensor cores (swapped operands) from 4 rows up,
// and from 2 rows for a B of 256 MB or more; the SIMT kernel below that,
// where one B vector feeds only one to three rows and the plain streaming
// kernel is faster (measured on GB300: 6.8 against 5.8 TB/s for one row of
// [8192, 28672], 5.2 against 2.0 TB/s for one row of [4096, 11008]).  The
// kernel-family override forces the SIMT kernel (variant 1) or the tensor
// cores (variant 2).
static bool skinny_m_on_tc(olc_dtype dt, const Problem& p) {
    if (!(dt == OLC_FLOAT16 || dt == OLC_BFLOAT16) || !tc_shape_ok(dt, p.N, p.K) || p.M > 16)
        return false;
    if (p.variant == 1) return false;
    if (p.variant == 2) return true;
    const double b_bytes = 2.0 * (double)p.K * (double)p.N * (double)p.items;
    return p.M >= 4 || (p.M >= 2 && b_bytes >= 256.0 * 1024 * 1024);
}

// E4M3FN / E5M2: the warp-MMA kernel from 4 rows, the SIMT kernel below
// (measured on GB300 for one [8192, 28672] B, TB/s, SIMT against MMA: 1 row
// 5.8 / 3.7, 2 rows 4.1 / 3.7, 4 rows 2.9 / 3.7, 16 rows 0.8 / 3.6); variant
// 1 forces the SIMT kernel, variant 2 the MMA kernel.
// E4M3FN / E5M2 on the tensor cores (variant 3): tcgen05 kind::f8f6f4 with
// swapped operands, B transposed in shared memory (fp8.cu)
static bool skinny_m_on_f8_tc(olc_dtype dt, const Problem& p) {
    return p.variant == 3 && f8_skinny_tc_ok(dt, p);
}

static bool skinny_m_on_f8_mma(olc_dtype dt, const Problem& p) {
    if (!(dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2) || p.M > 16 || p.N % 16 != 0) return false;
    if (skinny_m_on_f8_tc(dt, p)) return false;
    if (p.variant == 1) return false;
    if (p.variant == 2) return true;
    return p.M >= 4;
}

template <int FMT>
static int f8_mma_occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, skinny_m_f8_mma_kernel<FMT, 1>, kF8MmaWarps * 32, 0) !=
        cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    return n > 0 ? n : 4;   // no device visible: assume four resident blocks
}

static int skinny_m_simt_split(olc_dtype dt, const Problem& p, int sm_count);

int skinny_m_pick_split(olc_dtype dt, const Problem& p, int sm_count) {
    if (skinny_m_on_f8_tc(dt, p)) return f8_skinny_tc_pick(p, sm_count);
    return skinny_m_on_tc(dt, p) ? tc_skinny_m_pick(p, sm_count)
                                 : skinny_m_simt_split(dt, p, sm_count);
}

static int skinny_m_simt_split(olc_dtype dt, const Problem& p, int sm_count) {
    if (p.split_hint > 0) return (int)min64(p.split_hint, max64(1, p.K / 8));
    const bool mma = skinny_m_on_f8_mma(dt, p);
    const int64_t cols = mma ? kF8MmaCols : 32 * skinny_m_vec(dt, p.M);
    const int64_t groups = ceil_div(p.N, cols) * p.items;
    const int64_t slots = (int64_t)sm_count *
                          (mma ? (dt == OLC_FLOAT8E4M3FN ? f8_mma_occupancy<0>() : f8_mma_occupancy<1>())
                               : skinny_m_blocks_per_sm(dt, p.M));
    const int64_t eb = operand_bytes(dt);
    const int64_t acc = dt == OLC_DOUBLE ? 8 : 4;
    const int64_t rows = mma ? 16 : round_rows(p.M);
    const double stream_bytes = (double)p.K * p.N * eb * p.items;
    const int64_t smax = min64(64, max64(1, p.K / 256));
    int best = 1;
    double best_score = -1.0;
    for (int64_t s = 1; s <= smax; ++s) {
        const int64_t blocks = groups * s;
        const int64_t waves = ceil_div(blocks, slots);
        const double fill = (double)blocks / (double)(waves * slots);
        const double extra = s > 1 ? 2.0 * (double)s * rows * p.N * acc * p.items : 0.0;
        const double score = fill * stream_bytes / (stream_bytes + extra);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = (int)s;
        }
    }
    return best;
}

size_t skinny_m_partial_bytes(olc_dtype dt, const Problem& p, int ksplit, int sm_count) {
    if (skinny_m_on_f8_tc(dt, p)) return f8_skinny_tc_partial_bytes(p, ksplit);
    if (skinny_m_on_tc(dt, p)) return tc_skinny_m_partial_bytes(p, sm_count);
    if (skinny_m_on_f8_mma(dt, p))
        return (size_t)(ceil_div(p.N, kF8MmaCols) * p.items * ksplit * 16 * kF8MmaCols * 4);
    const int64_t acc = dt == OLC_DOUBLE ? 8 : 4;
    const int64_t entries = round_rows(p.M) * 32 * skinny_m_vec(dt, p.M);
    return (size_t)(skinny_m_col_groups(dt, p.M, p.N) * p.items * ksplit * entries * acc);
}

size_t skinny_m_counter_count(olc_dtype dt, const Problem& p, int ksplit, int sm_count) {
    if (skinny_m_on_f8_tc(dt, p)) return f8_skinny_tc_counter_count(p, ksplit);
    if (skinny_m_on_tc(dt, p)) return tc_skinny_m_counter_count(p, sm_count);
    if (skinny_m_on_f8_mma(dt, p)) return (size_t)(ceil_div(p.N, kF8MmaCols) * p.items);
    return (size_t)(skinny_m_col_groups(dt, p.M, p.N) * p.items);
}

template <typename T, int MR>
static cudaError_t launch_skinny_m_t(const Problem& p, int ksplit, const Workspace& ws,
                                     cudaStream_t s) {
    constexpr int VEC = SkinnyMVec<T, MR>::N;
    const int64_t groups = ceil_div(p.N, 32 * VEC);
    const int64_t kslice = ceil_div(ceil_div(p.K, ksplit), 8) * 8;
    const int64_t blocks = groups * ksplit * p.items;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (ksplit > 1 && (!ws.partials || !ws.counters)) return cudaErrorInvalidValue;
    // vector A loads (16 bytes; 8 for one-byte elements) need every A row
    // (and each operand item) aligned to the load
    const int64_t a_align = sizeof(T) == 1 ? 8 : 16;
    bool a_vec_ok = (p.K * (int64_t)sizeof(T)) % a_align == 0 &&
                    (reinterpret_cast<uintptr_t>(p.A) % a_align) == 0;
    for (int d = 0; d < p.map.rank; ++d)
        if ((p.map.a_stride[d] * (int64_t)sizeof(T)) % a_align != 0) a_vec_ok = false;
    skinny_m_kernel<T, MR><<<(unsigned)blocks, SkinnyMConfig<T, MR>::KW * 32, 0, s>>>(
        p, groups, ksplit, kslice, ws, a_vec_ok ? 1 : 0);
    return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_skinny_m_f8_mma(const Problem& p, int ksplit, const Workspace& ws, cudaStream_t s) {
    const int64_t groups = ceil_div(p.N, kF8MmaCols);
    const int64_t kslice = ceil_div(ceil_div(p.K, ksplit), 32) * 32;
    const int64_t blocks = groups * ksplit * p.items;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (ksplit > 1 && (!ws.partials || !ws.counters)) return cudaErrorInvalidValue;
    // 4-byte A loads need every A row (and each operand item) 4-byte aligned
    bool a_vec_ok = p.K % 4 == 0 && (reinterpret_cast<uintptr_t>(p.A) % 4) == 0;
    for (int d = 0; d < p.map.rank; ++d)
        if (p.map.a_stride[d] % 4 != 0) a_vec_ok = false;
    skinny_m_f8_mma_kernel<FMT, 1><<<(unsigned)blocks, kF8MmaWarps * 32, 0, s>>>(p, groups, ksplit, kslice, 0, ws,
                                                                             a_vec_ok ? 1 : 0);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SPLIT_K for E4M3FN / E5M2 products with small outputs (at most 32 rows and
// 128 columns, N a multiple of 16): the warp-MMA kernel above with one or two
// 16-row tiles, K cut into about one slice per SM, the partials summed in
// two fixed-order levels (skinny_m_finish_grouped).

constexpr int kF8SplitGroup = 16;   // slices per first-level group

bool f8_split_k_ok(olc_dtype dt, const Problem& p) {
    return (dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2) && p.M <= 32 && p.N % 16 == 0 && p.N <= 128 &&
           p.K > 0;
}

int f8_split_k_pick(const Problem& p, int sm_count) {
    const int64_t tiles = ceil_div(p.N, kF8MmaCols) * p.items;
    int64_t s = p.split_hint > 0 ? p.split_hint : ceil_div(sm_count, tiles);
    s = max64(1, min64(s, ceil_div(p.K, 32)));   // at least one 32-row chunk per slice
    const int64_t kslice = ceil_div(ceil_div(p.K, s), 32) * 32;
    return (int)ceil_div(p.K, kslice);           // no empty slices
}

size_t f8_split_k_partial_bytes(const Problem& p, int splits) {
    const int64_t tiles = ceil_div(p.N, kF8MmaCols) * p.items;
    return (size_t)(tiles * (splits + ceil_div(splits, kF8SplitGroup)) * 32 * kF8MmaCols * 4);
}

size_t f8_split_k_counter_count(const Problem& p, int splits) {
    const int64_t tiles = ceil_div(p.N, kF8MmaCols) * p.items;
    return (size_t)(tiles * (ceil_div(splits, kF8SplitGroup) + 1));
}

template <int FMT, int MT>
static cudaError_t launch_f8_split_t(const Problem& p, int splits, const Workspace& ws, cudaStream_t s) {
    const int64_t groups = ceil_div(p.N, kF8MmaCols);
    const int64_t kslice = ceil_div(ceil_div(p.K, splits), 32) * 32;
    const int64_t blocks = groups * splits * p.items;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (splits > 1 && (!ws.partials || !ws.counters || ws.partial_bytes < f8_split_k_partial_bytes(p, splits) ||
                       ws.counter_count < f8_split_k_counter_count(p, splits)))
        return cudaErrorInvalidValue;
    bool a_vec_ok = p.K % 4 == 0 && (reinterpret_cast<uintptr_t>(p.A) % 4) == 0;
    for (int d = 0; d < p.map.rank; ++d)
        if (p.map.a_stride[d] % 4 != 0) a_vec_ok = false;
    skinny_m_f8_mma_kernel<FMT, MT><<<(unsigned)blocks, kF8MmaWarps * 32, 0, s>>>(
        p, groups, splits, kslice, kF8SplitGroup, ws, a_vec_ok ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_f8_split_k(olc_dtype dt, const Problem& p, int splits, const Workspace& ws, cudaStream_t s) {
    if (!f8_split_k_ok(dt, p)) return cudaErrorInvalidValue;
    if (dt == OLC_FLOAT8E4M3FN)
        return p.M <= 16 ? launch_f8_split_t<0, 1>(p, splits, ws, s) : launch_f8_split_t<0, 2>(p, splits, ws, s);
    return p.M <= 16 ? launch_f8_split_t<1, 1>(p, splits, ws, s) : launch_f8_split_t<1, 2>(p, splits, ws, s);
}

cudaError_t launch_skinny_m(olc_dtype dt, const Problem& p, int ksplit, int sm_count,
                            const Workspace& ws, cudaStream_t s, const void* bt_ready) {
    if (skinny_m_on_tc(dt, p)) return launch_tc_skinny_m(dt, p, sm_count, ws, s);
    if (skinny_m_on_f8_tc(dt, p)) return launch_f8_skinny_tc(dt, p, ksplit, sm_count, ws, s, bt_ready);
    if (skinny_m_on_f8_mma(dt, p))
        return dt == OLC_FLOAT8E4M3FN ? launch_skinny_m_f8_mma<0>(p, ksplit, ws, s)
                                      : launch_skinny_m_f8_mma<1>(p, ksplit, ws, s);
    const int mr = round_rows(p.M);
    return dispatch_skinny_m(dt, cudaErrorInvalidValue, [&](auto tag) -> cudaError_t {
        using T = decltype(tag);
        switch (mr) {
            case 1: return launch_skinny_m_t<T, 1>(p, ksplit, ws, s);
            case 2: return launch_skinny_m_t<T, 2>(p, ksplit, ws, s);
            case 4: return launch_skinny_m_t<T, 4>(p, ksplit, ws, s);
            case 8: return launch_skinny_m_t<T, 8>(p, ksplit, ws, s);
            default: return launch_skinny_m_t<T, 16>(p, ksplit, ws, s);
        }
    });
}

// ===========================================================================
// SKINNY_N
//
// Block = 8 warps, each warp owns RW consecutive output rows; the block
// stages a KC-long chunk of B in shared memory, transposed (Bs[n][k]) and
// widened, so that lane l reading Bs[n][k0 + l] hits 32 distinct banks.  Lane
// l handles k = l, l + 32, ... of the chunk (coalesced A loads), keeps RW x NC
// partial sums and reuses each B value across the RW rows.  At the end the
// partial sums are reduced across the warp with shuffles (a fixed tree).

constexpr int kSkinnyNMax = 16;
int skinny_n_max_cols() { return kSkinnyNMax; }

template <typename T, int NC>
struct SkinnyNConfig {
    static constexpr int RW = 4;                       // rows per warp
    static constexpr int WARPS = 8;
    static constexpr int KC = (sizeof(typename Num<T>::acc_t) * NC * 1024 <= 64 * 1024) ? 1024 : 512;
};

template <typename T, int NC>
__global__ void __launch_bounds__(256)
skinny_n_kernel(Problem p, int64_t row_groups) {
    using acc_t = typename Num<T>::acc_t;
    using Cfg = SkinnyNConfig<T, NC>;
    constexpr int RW = Cfg::RW, KC = Cfg::KC, WARPS = Cfg::WARPS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    acc_t* Bs = reinterpret_cast<acc_t*>(smem_raw);   // [NC][KC]

    const int64_t item = blockIdx.x / row_groups;
    const int64_t rg = blockIdx.x % row_groups;
    int64_t a_off, b_off;
    batch_offsets(p.map, item, a_off, b_off);
    const T* __restrict__ A = static_cast<const T*>(p.A) + a_off;
    const T* __restrict__ B = static_cast<const T*>(p.B) + b_off;
    T* __restrict__ Y = static_cast<T*>(p.Y) + item * p.M * p.N;
    const int64_t M = p.M, N = p.N, K = p.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (rg * WARPS + warp) * RW;

    acc_t acc[RW][NC];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int n = 0; n < NC; ++n) acc[r][n] = acc_t(0);

    for (int64_t kc = 0; kc < K; kc += KC) {
        const int klen = (int)min64(KC, K - kc);
        __syncthreads();
        for (int e = threadIdx.x; e < KC * NC; e += blockDim.x) {
            const int k = e / NC, n = e % NC;
            Bs[n * KC + k] = (k < klen && n < N) ? Num<T>::to_acc(B[(kc + k) * N + n]) : acc_t(0);
        }
        __syncthreads();
        for (int k = lane; k < klen; k += 32) {
            acc_t a[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r)
                a[r] = (row0 + r < M) ? Num<T>::to_acc(__ldg(A + (row0 + r) * K + kc + k)) : acc_t(0);
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const acc_t b = Bs[n * KC + k];
#pragma unroll
                for (int r = 0; r < RW; ++r) acc[r][n] = fma(a[r], b, acc[r][n]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            acc_t v = acc[r][n];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r][n] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            if (row0 + r >= M) continue;
#pragma unroll
            for (int n = 0; n < NC; ++n)
                if (n < N)
                    Y[(row0 + r) * N + n] =
                        Num<T>::from_acc(apply_epilogue<T>(p.epi, acc[r][n], row0 + r, n, Y + (row0 + r) * N + n));
        }
    }
}

template <typename T, int NC>
static cudaError_t launch_skinny_n_t(const Problem& p, cudaStream_t s) {
    using Cfg = SkinnyNConfig<T, NC>;
    const int64_t rows_per_block = Cfg::RW * Cfg::WARPS;
    const int64_t groups = ceil_div(p.M, rows_per_block);
    const int64_t blocks = groups * p.items;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(typename Num<T>::acc_t) * NC * Cfg::KC;
    if (smem > 48 * 1024) {
        const cudaError_t attr =
            set_smem_limit(reinterpret_cast<const void*>(skinny_n_kernel<T, NC>), (int)smem);
        if (attr != cudaSuccess) return attr;
    }
    skinny_n_kernel<T, NC><<<(unsigned)blocks, 256, smem, s>>>(p, groups);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SKINNY_N for FLOAT16 / BFLOAT16: A streamed with 16-byte loads straight
// into registers, the products on the tensor cores with mma.sync.m16n8k16
// (float32 accumulation), B in shared memory.
//
// A unit is 16 rows of A (all K); one persistent block per SM owns every
// gridDim-th unit, and its 16 warps each take one sixteenth of K of every
// unit.  The warps run independently through the block's units: a warp
// writes its 16 x 8 (or 16 x 16) float32 partial tile to one of kSnSlots
// shared-memory slots and counts itself in; the sixteenth warp to arrive
// sums the sixteen partials in K-range order (a fixed order: the result does
// not depend on timing), applies the epilogue and stores the rows, then
// frees the slot.  No block-wide barrier stops the loads, so while some
// warps reduce or wait, the others keep their 16-byte loads in flight.
// Register loads are used instead of TMA tiles: 512 threads per SM with
// sixteen 16-byte loads each stream A at close to the HBM rate, where 2-D
// tensor boxes of 128-byte rows did not.
//
// Thread (g = lane / 4, t = lane % 4) loads A[row g][k0 + 8t .. 8t + 7] and
// A[row g + 8][...] (16 bytes each) for every 32-wide K chunk k0.  The MMA's
// K positions are relabelled so that these are exactly the thread's A
// fragment of two m16n8k16 products: the first takes physical k = 8t + {0,
// 1} and 8t + {2, 3} for its logical k = 2t + {0, 1} and 2t + 8 + {0, 1},
// the second 8t + {4 .. 7}.  Relabelling the terms of a dot product does
// not change which products are summed, so each output is still the full
// dot product.  The B fragments under the same relabelling come from one
// ldmatrix.x4.trans per chunk: B sits in shared memory as 16-byte rows (8
// columns, one plane per 8 columns), and the lanes hand ldmatrix the row
// addresses in the relabelled order (matrix i, row r: k = k0 + 8 (r / 2) +
// 2i + r % 2), so the transposed 8 x 8 matrices land as exactly the b
// registers of the two products.  Rows are placed with an XOR swizzle (row
// k at 16-byte slot k ^ (((k >> 3) & 3) << 1)) so that the eight rows of
// each matrix fall in eight different bank groups.
//
// E4M3FN / E5M2 operands use the same streaming and the same register
// assignment with mma.sync.m16n8k32 (8-bit operands, float32 accumulation,
// FLOAT output): a chunk is 64 K positions (the same 64 bytes of each row),
// thread t's 16 bytes hold k0 + 16t .. 16t + 15, and the first product takes
// 16t + {0..3} and 16t + {4..7} for its logical K positions 4t + {0..3} and
// 16 + 4t + {0..3}, the second 16t + {8..15}.  B is staged transposed, one
// row of K bytes per column (rows padded to 64 bytes past a multiple of 128,
// so that the two columns a quarter-warp reads fall in different banks), and
// a thread's two B fragments of an 8-column block are one 16-byte shared
// load at its column and k0 + 16t.

constexpr int kSnWarps = 16;
constexpr int kSnSlots = 4;

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, bool bf16) {
    if (bf16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

__device__ __forceinline__ uint4 ldmatrix_x4_trans(uint32_t addr) {
    uint4 r;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// 16-byte slot of B row k in its plane
__device__ __forceinline__ int64_t sn_slot(int64_t k) { return k ^ (((k >> 3) & 3) << 1); }

// K per warp (whole chunks of ck elements, 64 bytes of a row) and the rows
// of a B plane (every warp's range; rows at or past K hold zeros).
static int64_t sn_k_per_warp(int64_t K, int ck) { return ceil_div(ceil_div(K, kSnWarps), ck) * ck; }
static int64_t sn_rows(int64_t K, int ck) { return sn_k_per_warp(K, ck) * kSnWarps; }
// shared-memory bytes of B: 16-byte rows per 8-column plane (16-bit types),
// or one transposed row of K bytes (+ 64 bytes) per column (8-bit types)
static int64_t sn_b_bytes(int eb, int nb, int64_t K) {
    return eb == 1 ? (int64_t)nb * 8 * (sn_rows(K, 64) + 64) : (int64_t)nb * sn_rows(K, 32) * 16;
}

template <int NB>
struct SnShared {
    float red[kSnSlots][kSnWarps][16][NB * 8 + 1];   // partial tiles (+1: no bank conflicts)
    int arrived[kSnSlots];                          // warps counted into the slot's unit
    int uses[kSnSlots];                             // reductions completed in the slot
    int abort;
};

template <typename T, int NB>
__global__ void __launch_bounds__(kSnWarps * 32, 1)
skinny_n_mma_kernel(Problem p, int64_t units, int kw, int64_t rows, unsigned int* err) {
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr bool F8 = sizeof(T) == 1;
    using out_t = typename Num<T>::out_t;
    constexpr int EB = (int)sizeof(T);
    constexpr int CK = 64 / EB;                            // K positions per chunk
    constexpr int R = 8;                                   // K chunks in flight per thread
    // 16-bit types: [NB planes][rows] 16-byte B rows; 8-bit: [NB * 8 columns][rows + 64] bytes
    extern __shared__ __align__(16) uint4 bs[];
    __shared__ SnShared<NB> sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t M = p.M, N = p.N, K = p.K;
    // K range of this warp: rotated by the block index, so that at the
    // start the blocks ask L2 for different lines of B instead of all for
    // the same ones (the partials are still summed in K-range order)
    const int krange = (warp + (int)(blockIdx.x % kSnWarps)) % kSnWarps;
    const int64_t kbeg = (int64_t)krange * kw;
    const unsigned char* A = static_cast<const unsigned char*>(p.A);

    // This warp's work is one sequence of 32-wide K chunks: chunk c of its K
    // range for each of the block's units in turn.  A ring of R register
    // slots keeps R chunks (2 x 16 bytes per thread each) in flight: chunk
    // i + R is requested as soon as chunk i has been multiplied.
    const int cpu = kw / CK;                               // chunks per unit
    const int my_units = (int)((units - blockIdx.x + gridDim.x - 1) / gridDim.x);
    // the next chunk to request: unit index (within this block) and chunk
    int lu = 0, lc = 0;
    auto load = [&](uint4& va, uint4& vb) {
        va = make_uint4(0u, 0u, 0u, 0u);
        vb = va;
        if (lu < my_units) {
            const int64_t r0 = (blockIdx.x + (int64_t)lu * gridDim.x) * 16;
            // K is a multiple of 16 bytes: a 16-byte piece starting below K is whole
            const int64_t k = kbeg + lc * CK + (CK / 4) * t;
            const int64_t ra = r0 + g, rb = r0 + g + 8;
            if (k < K && ra < M) va = __ldcs(reinterpret_cast<const uint4*>(A + (ra * K + k) * EB));
            if (k < K && rb < M) vb = __ldcs(reinterpret_cast<const uint4*>(A + (rb * K + k) * EB));
        }
        if (++lc == cpu) { lc = 0; ++lu; }
    };
    if (threadIdx.x < kSnSlots) {
        sh.arrived[threadIdx.x] = 0;
        sh.uses[threadIdx.x] = 0;
    }
    if (threadIdx.x == 0) sh.abort = 0;
    __syncthreads();   // slot counters initialised before any warp arrives
    grid_dependency_wait();
    grid_launch_dependents();

    // Each warp stages only the B rows of its own K range, so it never waits
    // for the others.  With N == 8 or 16 every 16-byte vector of B is one
    // row of one plane and is stored as it is; other N are padded to 8
    // columns element by element.  Rows at or past K are zero.
    const int64_t rstride = rows + 64;                    // 8-bit types: bytes per transposed row
    {
        const int64_t kend = min64(K, kbeg + kw);
        if constexpr (F8) {
            const unsigned char* B = static_cast<const unsigned char*>(p.B);
            unsigned char* bt = reinterpret_cast<unsigned char*>(bs);
            for (int v = lane; v < kw * NB * 8; v += 32) {
                const int n = v % (NB * 8);
                const int64_t k = kbeg + v / (NB * 8);
                bt[n * rstride + k] = (k < kend && n < N) ? __ldg(B + k * N + n) : (unsigned char)0;
            }
        } else if (N == 8 * NB) {
            const uint4* B4 = static_cast<const uint4*>(p.B);
            for (int v0 = lane; v0 < kw * NB; v0 += 4 * 32) {
                uint4 w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int v = v0 + q * 32;
                    const int64_t k = kbeg + v / NB;
                    w[q] = (v < kw * NB && k < kend) ? __ldg(B4 + k * NB + v % NB)
                                                     : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int v = v0 + q * 32;
                    if (v < kw * NB) bs[(v % NB) * rows + sn_slot(kbeg + v / NB)] = w[q];
                }
            }
        } else {
            const unsigned short* B = static_cast<const unsigned short*>(p.B);
            for (int v = lane; v < kw * NB; v += 32) {
                const int j = v % NB;
                const int64_t k = kbeg + v / NB;
                uint32_t h[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int64_t n = j * 8 + c;
                    const uint32_t e = (k < kend && n < N) ? (uint32_t)B[k * N + n] : 0u;
                    h[c >> 1] |= e << (16 * (c & 1));
                }
                bs[j * rows + sn_slot(k)] = make_uint4(h[0], h[1], h[2], h[3]);
            }
        }
        __syncwarp();
    }
    uint4 va[R], vb[R];
#pragma unroll
    for (int q = 0; q < R; ++q) load(va[q], vb[q]);

    // ldmatrix row address of this lane for chunk base k0: matrix i = lane /
    // 8, row r = lane % 8 -> k = k0 + 8 (r / 2) + 2 i + r % 2
    const int mi = lane >> 3, mr = lane & 7;
    const int koff = 8 * (mr >> 1) + 2 * mi + (mr & 1);
    const uint32_t bs_base = static_cast<uint32_t>(__cvta_generic_to_shared(bs));

    out_t* Y = static_cast<out_t*>(p.Y);
    volatile int* uses = sh.uses;
    volatile int* abort_flag = &sh.abort;
    // two accumulator chains per n-block (the two MMAs of a chunk), summed
    // when the unit is done
    float d0[NB][4], d1[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) d0[j][e] = d1[j][e] = 0.f;

    // one unit's partial tile -> its slot; the sixteenth warp reduces
    auto flush = [&](int ui) -> bool {
        const int64_t r0 = ((int64_t)blockIdx.x + (int64_t)ui * gridDim.x) * 16;
        const int slot = (int)(ui % kSnSlots);
        const int use = (int)(ui / kSnSlots);
        int ok = 1;
        if (lane == 0 && uses[slot] != use) {              // bounded wait for the slot
            const uint64_t t0 = globaltimer_ns();
            while (uses[slot] != use) {
                if (*abort_flag || globaltimer_ns() - t0 > 2000000000ull) {
                    if (!*abort_flag) {
                        *abort_flag = 1;
                        raise_device_error(err, kErrWaitTimeout);
                    }
                    ok = 0;
                    break;
                }
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        // row g: elements 0, 1 (columns 2t, 2t + 1); row g + 8: elements 2, 3;
        // partials are filed by K range
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            sh.red[slot][krange][g][j * 8 + 2 * t] = d0[j][0] + d1[j][0];
            sh.red[slot][krange][g][j * 8 + 2 * t + 1] = d0[j][1] + d1[j][1];
            sh.red[slot][krange][g + 8][j * 8 + 2 * t] = d0[j][2] + d1[j][2];
            sh.red[slot][krange][g + 8][j * 8 + 2 * t + 1] = d0[j][3] + d1[j][3];
#pragma unroll
            for (int e = 0; e < 4; ++e) d0[j][e] = d1[j][e] = 0.f;
        }
        __threadfence_block();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&sh.arrived[slot], 1) == kSnWarps - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            for (int e = lane; e < 16 * NB * 8; e += 32) {
                const int r = e / (NB * 8), c = e % (NB * 8);
                const int64_t row = r0 + r;
                if (row >= M || c >= N) continue;
                float v = sh.red[slot][0][r][c];
#pragma unroll
                for (int w = 1; w < kSnWarps; ++w) v += sh.red[slot][w][r][c];
                Y[row * N + c] = Num<T>::from_acc(apply_epilogue<out_t>(p.epi, v, row, c, Y + row * N + c));
            }
            __syncwarp();
            if (lane == 0) {
                sh.arrived[slot] = 0;
                __threadfence_block();
                uses[slot] = use + 1;
            }
        }
        return true;
    };

    // the chunk being multiplied: unit index (within this block) and chunk
    int cu = 0, cc = 0;
    while (cu < my_units) {
#pragma unroll
        for (int q = 0; q < R; ++q) {
            if (cu >= my_units) break;
            if constexpr (F8) {
                const uint32_t kb = (uint32_t)(kbeg + cc * CK + 16 * t);
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const uint4 b = *reinterpret_cast<const uint4*>(
                        reinterpret_cast<const unsigned char*>(bs) + (j * 8 + g) * rstride + kb);
                    const uint32_t a0[4] = {va[q].x, vb[q].x, va[q].y, vb[q].y};
                    const uint32_t a1[4] = {va[q].z, vb[q].z, va[q].w, vb[q].w};
                    mma_f8_m16n8k32<T::kFormat>(d0[j], a0, b.x, b.y);
                    mma_f8_m16n8k32<T::kFormat>(d1[j], a1, b.z, b.w);
                }
            } else {
                const int64_t krow = sn_slot(kbeg + cc * 32 + koff);
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const uint4 b = ldmatrix_x4_trans(bs_base + (uint32_t)((j * rows + krow) * 16));
                    mma_16816(d0[j], va[q].x, vb[q].x, va[q].y, vb[q].y, b.x, b.y, BF16);
                    mma_16816(d1[j], va[q].z, vb[q].z, va[q].w, vb[q].w, b.z, b.w, BF16);
                }
            }
            load(va[q], vb[q]);
            if (++cc == cpu) {
                if (!flush(cu)) return;
                cc = 0;
                ++cu;
            }
        }
    }
}

// Largest B (bytes, 16-byte rows per 8 columns) the streaming kernel keeps
// in shared memory (one block per SM, next to the partial-tile slots).
constexpr int64_t kSnMaxBtBytes = 150 * 1024;
static_assert(kSnMaxBtBytes + sizeof(SnShared<2>) <= 227 * 1024, "shared memory of one block");

bool skinny_n_mma_ok(olc_dtype dt, const Problem& p) {
    const bool f8 = dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2;
    if (dt != OLC_FLOAT16 && dt != OLC_BFLOAT16 && !f8) return false;
    // 16-byte pieces of A rows: K a multiple of 8 (16-bit) or 16 (8-bit)
    if (p.N > 16 || (p.K % (f8 ? 16 : 8)) != 0) return false;
    // one B for every unit: a single item, or items folded into rows
    if (p.items != 1) return false;
    // above 8 columns the tcgen05 16-column kernel is faster for 16-bit
    // types (two mma.sync per 8 columns cost more than one 128 x 16 tcgen05
    // MMA); 8-bit types have no such kernel
    if (!f8 && p.N > 8 && p.variant != 2) return false;
    const int nb = p.N <= 8 ? 1 : 2;                       // 8-column planes
    return sn_b_bytes(f8 ? 1 : 2, nb, p.K) <= kSnMaxBtBytes;
}

bool skinny_n_f8_ok(olc_dtype dt, const Problem& p) {
    return (dt == OLC_FLOAT8E4M3FN || dt == OLC_FLOAT8E5M2) && skinny_n_mma_ok(dt, p);
}

template <typename T, int NB>
static cudaError_t launch_skinny_n_mma_t(const Problem& p, int sm_count, cudaStream_t s) {
    constexpr int CK = 64 / (int)sizeof(T);
    const int64_t units = ceil_div(p.M, 16);
    const int kw = (int)sn_k_per_warp(p.K, CK);
    const int64_t rows = sn_rows(p.K, CK);
    const size_t smem = (size_t)sn_b_bytes((int)sizeof(T), NB, p.K);
    const cudaError_t attr = set_smem_limit(reinterpret_cast<const void*>(skinny_n_mma_kernel<T, NB>),
                                            (int)kSnMaxBtBytes);
    if (attr != cudaSuccess) return attr;
    const int64_t grid = min64(units, (int64_t)sm_count);
    return launch_pdl(skinny_n_mma_kernel<T, NB>, dim3((unsigned)grid), dim3(kSnWarps * 32), smem, s,
                      p, units, kw, rows, device_error_word());
}

static cudaError_t launch_skinny_n_mma(olc_dtype dt, const Problem& p, int sm_count,
                                       cudaStream_t s) {
    if (dt == OLC_FLOAT8E4M3FN)
        return p.N <= 8 ? launch_skinny_n_mma_t<F8<0>, 1>(p, sm_count, s)
                        : launch_skinny_n_mma_t<F8<0>, 2>(p, sm_count, s);
    if (dt == OLC_FLOAT8E5M2)
        return p.N <= 8 ? launch_skinny_n_mma_t<F8<1>, 1>(p, sm_count, s)
                        : launch_skinny_n_mma_t<F8<1>, 2>(p, sm_count, s);
    if (dt == OLC_FLOAT16)
        return p.N <= 8 ? launch_skinny_n_mma_t<__half, 1>(p, sm_count, s)
                        : launch_skinny_n_mma_t<__half, 2>(p, sm_count, s);
    return p.N <= 8 ? launch_skinny_n_mma_t<__nv_bfloat16, 1>(p, sm_count, s)
                    : launch_skinny_n_mma_t<__nv_bfloat16, 2>(p, sm_count, s);
}

static bool skinny_n_on_tc(olc_dtype dt, const Problem& p) {
    return (dt == OLC_FLOAT16 || dt == OLC_BFLOAT16) && tc_shape_ok(dt, p.N, p.K);
}

size_t skinny_n_partial_bytes(olc_dtype dt, const Problem& p, int sm_count) {
    return skinny_n_on_tc(dt, p) ? tc_skinny_n_partial_bytes(p, sm_count) : 0;
}

size_t skinny_n_counter_count(olc_dtype dt, const Problem& p, int sm_count) {
    return skinny_n_on_tc(dt, p) ? tc_skinny_n_counter_count(p, sm_count) : 0;
}

cudaError_t launch_skinny_n(olc_dtype dt, const Problem& p, int sm_count, const Workspace& ws,
                            cudaStream_t s) {
    // FLOAT16 / BFLOAT16 with 16-byte row strides: stream A through the
    // tensor cores with 16-column tiles (8 FMAs per A element would need most
    // of the SIMT FMA rate at full HBM bandwidth)
    if (skinny_n_f8_ok(dt, p)) return launch_skinny_n_mma(dt, p, sm_count, s);   // 8-bit: the only kernel
    if (p.variant != 1 && skinny_n_mma_ok(dt, p)) return launch_skinny_n_mma(dt, p, sm_count, s);
    if (skinny_n_on_tc(dt, p)) return launch_skinny_n_tc(dt, p, sm_count, ws, s);
    return dispatch_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        if (p.N <= 1) return launch_skinny_n_t<T, 1>(p, s);
        if (p.N <= 2) return launch_skinny_n_t<T, 2>(p, s);
        if (p.N <= 4) return launch_skinny_n_t<T, 4>(p, s);
        if (p.N <= 8) return launch_skinny_n_t<T, 8>(p, s);
        return launch_skinny_n_t<T, 16>(p, s);
    });
}

}  // namespace olc
