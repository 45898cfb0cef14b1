// Device helpers shared by the kernel files: element types, the batch map
// walk, and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "olc_internal.h"

namespace olc {

// Element traits: accumulator type and the load / narrowing store.  FP16 and
// BF16 accumulate in float32 and narrow once with round-to-nearest-even.
template <typename T>
struct Num;

template <>
struct Num<float> {
    using acc_t = float;
    using out_t = float;
    static __device__ __forceinline__ float to_acc(float v) { return v; }
    static __device__ __forceinline__ float from_acc(float v) { return v; }
};
template <>
struct Num<double> {
    using acc_t = double;
    using out_t = double;
    static __device__ __forceinline__ double to_acc(double v) { return v; }
    static __device__ __forceinline__ double from_acc(double v) { return v; }
};
template <>
struct Num<__half> {
    using acc_t = float;
    using out_t = __half;
    static __device__ __forceinline__ float to_acc(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_acc(float v) { return __float2half_rn(v); }
};
template <>
struct Num<__nv_bfloat16> {
    using acc_t = float;
    using out_t = __nv_bfloat16;
    static __device__ __forceinline__ float to_acc(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_acc(float v) { return __float2bfloat16_rn(v); }
};

// GELU in float32: y Phi(y) = y / 2 (1 + erf(z)), z = y / sqrt 2, with
// erfc(|z|) from the rational approximation of Abramowitz and Stegun,
// Handbook of Mathematical Functions, formula 7.1.26 (absolute error at
// most 1.5e-7): erfc(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
// t = 1 / (1 + p x), x >= 0.  Then 1 + erf(z) is 2 - erfc(|z|) for z >= 0 and
// erfc(|z|) for z < 0, which avoids cancellation on the negative side.  The
// body is short because the epilogue inlines it once per accumulator
// register of its unrolled store loop.
__device__ __forceinline__ float gelu_f32(float y) {
    const float z = y * 0.70710678118654752f;
    const float az = fabsf(z);
    const float t = __fdividef(1.0f, fmaf(0.3275911f, az, 1.0f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    const float c = q * t * __expf(-az * az);            // erfc(|z|)
    const float one_plus_erf = z >= 0.f ? 2.0f - c : c;  // NaN takes the second arm
    return 0.5f * y * one_plus_erf;
}

// The fused epilogue's activation, in the accumulator type.
__device__ __forceinline__ float activate(int act, float y) {
    if (act == OLC_ACT_RELU) return y < 0.f ? 0.f : y;    // NaN fails the test: stays NaN
    if (act == OLC_ACT_GELU) return gelu_f32(y);
    return y;
}
__device__ __forceinline__ double activate(int act, double y) {
    if (act == OLC_ACT_RELU) return y < 0.0 ? 0.0 : y;
    // 1 + erf(z) = erfc(-z): no cancellation for negative y
    if (act == OLC_ACT_GELU) return 0.5 * y * erfc(-y * 0.70710678118654752440);
    return y;
}

// Where the residual of the output element at y sits (R has Y's layout).
template <typename T>
__device__ __forceinline__ const T* residual_at(const Epilogue& e, const T* y) {
    return reinterpret_cast<const T*>(reinterpret_cast<const unsigned char*>(y) + e.r_delta);
}

// The epilogue on one accumulator of output (i, j) (within its item), to be
// stored at y: alpha * acc + beta * C, plus the residual, then the
// activation.  Each product and sum is rounded separately (no contraction),
// in the accumulator type.
template <typename T>
__device__ __forceinline__ typename Num<T>::acc_t apply_epilogue(const Epilogue& e,
                                                                 typename Num<T>::acc_t acc,
                                                                 int64_t i, int64_t j,
                                                                 const T* y) {
    using acc_t = typename Num<T>::acc_t;
    if (e.mode == 0) return acc;
    if constexpr (sizeof(acc_t) == 8) {
        double v = __dmul_rn(e.alpha_d, acc);
        if (e.C) {
            const double c = Num<T>::to_acc(static_cast<const T*>(e.C)[i * e.c_rs + j * e.c_cs]);
            v = __dadd_rn(v, __dmul_rn(e.beta_d, c));
        }
        if (e.R) v = __dadd_rn(v, Num<T>::to_acc(*residual_at(e, y)));
        return activate(e.act, v);
    } else {
        float v = __fmul_rn(e.alpha_f, acc);
        if (e.C) {
            const float c = Num<T>::to_acc(__ldg(static_cast<const T*>(e.C) + i * e.c_rs + j * e.c_cs));
            v = __fadd_rn(v, __fmul_rn(e.beta_f, c));
        }
        if (e.R) v = __fadd_rn(v, Num<T>::to_acc(__ldg(residual_at(e, y))));
        return activate(e.act, v);
    }
}

// 8-bit float operands, decoded from the format fields (exact in float32).
// E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is
// NaN, no infinities.  E5M2: sign, 5 exponent bits (bias 15), 2 mantissa
// bits; exponent 31 holds infinities and NaNs.
__device__ __forceinline__ float fp8_e4m3_to_f32(uint32_t b) {
    const uint32_t sign = (b & 0x80u) << 24;
    const uint32_t e = (b >> 3) & 0xFu, m = b & 0x7u;
    if ((b & 0x7Fu) == 0x7Fu) return __uint_as_float(sign | 0x7FC00000u);
    const float mag = e == 0 ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return __uint_as_float(__float_as_uint(mag) | sign);
}
__device__ __forceinline__ float fp8_e5m2_to_f32(uint32_t b) {
    const uint32_t sign = (b & 0x80u) << 24;
    const uint32_t e = (b >> 2) & 0x1Fu, m = b & 0x3u;
    if (e == 31u) return __uint_as_float(sign | (m == 0 ? 0x7F800000u : 0x7FC00000u));
    const float mag = e == 0 ? (float)m * 0x1p-16f : __uint_as_float(((e + 112u) << 23) | (m << 21));
    return __uint_as_float(__float_as_uint(mag) | sign);
}

// FNUZ variants: exponent bias one larger (8 / 16), no infinities, no
// negative zero, 0x80 the only NaN
__device__ __forceinline__ float fp8_e4m3fnuz_to_f32(uint32_t b) {
    if (b == 0x80u) return __uint_as_float(0x7FC00000u);
    const uint32_t sign = (b & 0x80u) << 24;
    const uint32_t e = (b >> 3) & 0xFu, m = b & 0x7u;
    const float mag = e == 0 ? (float)m * 0x1p-10f : __uint_as_float(((e + 119u) << 23) | (m << 20));
    return __uint_as_float(__float_as_uint(mag) | sign);
}
__device__ __forceinline__ float fp8_e5m2fnuz_to_f32(uint32_t b) {
    if (b == 0x80u) return __uint_as_float(0x7FC00000u);
    const uint32_t sign = (b & 0x80u) << 24;
    const uint32_t e = (b >> 2) & 0x1Fu, m = b & 0x3u;
    const float mag = e == 0 ? (float)m * 0x1p-17f : __uint_as_float(((e + 111u) << 23) | (m << 21));
    return __uint_as_float(__float_as_uint(mag) | sign);
}

// One 8-bit float operand element of format FMT (0 E4M3FN, 1 E5M2,
// 2 E4M3FNUZ, 3 E5M2FNUZ): decoded exactly to float32, accumulated in
// float32, and the output is float32 (no narrowing).
template <int FMT>
struct F8 {
    static constexpr int kFormat = FMT;
    unsigned char bits;
};
template <int FMT>
__device__ __forceinline__ float fp8_decode(uint32_t b) {
    if constexpr (FMT == 0) return fp8_e4m3_to_f32(b);
    else if constexpr (FMT == 1) return fp8_e5m2_to_f32(b);
    else if constexpr (FMT == 2) return fp8_e4m3fnuz_to_f32(b);
    else return fp8_e5m2fnuz_to_f32(b);
}
template <int FMT>
struct Num<F8<FMT>> {
    using acc_t = float;
    using out_t = float;
    static __device__ __forceinline__ float to_acc(F8<FMT> v) { return fp8_decode<FMT>(v.bits); }
    static __device__ __forceinline__ float from_acc(float v) { return v; }
};

// 8-bit float elements packed in WORDS 32-bit words (element i in byte i of
// the little-endian sequence) to float32.  E4M3FN and E5M2 go through the hardware pair conversion to half
// precision, which holds every value of both formats exactly, then to
// float32; the FNUZ formats are decoded from their fields.
template <int FMT, int WORDS>
__device__ __forceinline__ void fp8_decode_words(const uint32_t (&w)[WORDS], float (&out)[4 * WORDS]) {
#pragma unroll
    for (int q = 0; q < WORDS; ++q) {
        if constexpr (FMT <= 1) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
                    (__nv_fp8x2_storage_t)((w[q] >> (16 * h)) & 0xFFFFu), FMT == 0 ? __NV_E4M3 : __NV_E5M2);
                __half_raw lo, hi;
                lo.x = r.x;
                hi.x = r.y;
                out[4 * q + 2 * h] = __half2float(__half(lo));
                out[4 * q + 2 * h + 1] = __half2float(__half(hi));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) out[4 * q + i] = fp8_decode<FMT>((w[q] >> (8 * i)) & 0xFFu);
        }
    }
}
// Paired FP32 multiply-add (Blackwell fma.rn.f32x2): d = a * b + d on two
// lanes of packed floats, one issue slot for two FMAs.
__device__ __forceinline__ unsigned long long pack_f2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f2(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma_f2(unsigned long long& d, unsigned long long a,
                                       unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// one element through the read-only path (8-bit float elements as bytes)
template <typename T>
__device__ __forceinline__ T ldg_elem(const T* p) {
    return __ldg(p);
}
template <int FMT>
__device__ __forceinline__ F8<FMT> ldg_elem(const F8<FMT>* p) {
    return F8<FMT>{__ldg(reinterpret_cast<const unsigned char*>(p))};
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Operand element offsets of output batch item z.
__device__ __forceinline__ void batch_offsets(const BatchMap& m, int64_t z, int64_t& a_off,
                                              int64_t& b_off) {
    a_off = 0;
    b_off = 0;
#pragma unroll 1
    for (int d = m.rank - 1; d >= 0; --d) {
        const int64_t e = m.dims[d];
        const int64_t i = z % e;
        z /= e;
        a_off += i * m.a_stride[d];
        b_off += i * m.b_stride[d];
    }
}

// Device error word: bit flags set by kernels whose bounded waits ran out.
// Kernels receive its address (device_error_word()) as an argument.
constexpr unsigned int kErrWaitTimeout = 1u;

__device__ __forceinline__ void raise_device_error(unsigned int* word, unsigned int bits) {
    if (word) atomicOr(word, bits);
}

template <typename F>
inline cudaError_t dispatch_dtype(olc_dtype dt, F&& f) {
    switch (dt) {
        case OLC_FLOAT: return f(float{});
        case OLC_DOUBLE: return f(double{});
        case OLC_FLOAT16: return f(__half{});
        case OLC_BFLOAT16: return f(__nv_bfloat16{});
        default: break;   // 8-bit float types have kernels of their own
    }
    return cudaErrorInvalidValue;
}

template <typename F>
inline int dispatch_int(olc_dtype dt, F&& f) {
    switch (dt) {
        case OLC_FLOAT: return f(float{});
        case OLC_DOUBLE: return f(double{});
        case OLC_FLOAT16: return f(__half{});
        case OLC_BFLOAT16: return f(__nv_bfloat16{});
        default: break;
    }
    return 0;
}

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per (kernel, device): the attribute belongs to the device's context, so a
// process that launches on several devices sets it on each of them.
inline cudaError_t set_smem_limit(const void* kernel, int bytes) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static std::vector<std::pair<const void*, uint64_t>> done;   // kernel -> device mask
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < kMaxDevices ? (1ull << dev) : 0ull;
    std::lock_guard<std::mutex> lock(mu);
    uint64_t* mask = nullptr;
    for (auto& d : done)
        if (d.first == kernel) {
            mask = &d.second;
            break;
        }
    if (mask && bit && (*mask & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (!mask) {
        done.emplace_back(kernel, 0ull);
        mask = &done.back().second;
    }
    *mask |= bit;
    return cudaSuccess;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the previous kernel in the stream is still finishing; it calls
// grid_dependency_wait() before its first access to global memory (the wait
// returns once that kernel has completed and its writes are visible; without
// the launch attribute it returns at once) and grid_launch_dependents() to
// let the next such launch start its own prologue.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace olc
