// Arithmetic-rate probe for the FP32 / FP64 rooflines.
//
// The FLOAT and DOUBLE kernels are bound by the FMA pipes, not by memory or
// the tensor cores (FP32 and FP64 MatMul keep native precision: no TF32).
// Their roofline peak is derived from unit counts and the clock (152 SMs x
// 128 FP32 lanes x 2 flop x clock; 152 SMs x 4 FP64 flop x clock).  This
// probe measures what the pipes actually deliver on the device at hand: every
// thread of SMs x 4 blocks of 256 threads runs 8 independent FMA chains
// acc = a * b + acc (the accumulator as the addend, as in a GEMM),
// unrolled 8 deep so that loop control takes few issue slots (no memory
// traffic, no dependency stalls once all warps are resident); one launch of
// the same length warms up, and the elapsed time of a second gives flop/s.
// Kinds:
//   0  paired FP32 FMA (fma.rn.f32x2: two FMAs per issue)
//   1  scalar FP32 FMA (fma.rn.f32)
//   2  FP64 FMA (fma.rn.f64)
//   3  FP64 tensor-core MMA (mma.sync m8n8k4 .f64, 256 FMAs per warp issue)
#include "common.cuh"

namespace olc {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeBlocksPerSm = 4;
constexpr int kChains = 8;

// written only when a result equals an impossible value, so the compiler
// keeps every chain without a memory store per thread
__device__ float g_probe_sink_f;
__device__ double g_probe_sink_d;

__global__ void __launch_bounds__(kProbeThreads) probe_ffma2(long long iters, float seed) {
    unsigned long long acc[kChains];
    const float t = seed + threadIdx.x * 1e-7f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = pack_f2(t + c, t - c);
    const unsigned long long a = pack_f2(0.999999f, 0.999998f);
    const unsigned long long b = pack_f2(1e-7f, 2e-7f);
#pragma unroll 8
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc[c]) : "l"(a), "l"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        float lo, hi;
        unpack_f2(acc[c], lo, hi);
        s += lo + hi;
    }
    if (s == 1234567.0f) g_probe_sink_f = s;
}

__global__ void __launch_bounds__(kProbeThreads) probe_ffma(long long iters, float seed) {
    float acc[kChains];
    const float t = seed + threadIdx.x * 1e-7f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = t + c;
#pragma unroll 8
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("fma.rn.f32 %0, %1, %2, %0;" : "+f"(acc[c]) : "f"(0.999999f), "f"(1e-7f));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    if (s == 1234567.0f) g_probe_sink_f = s;
}

__global__ void __launch_bounds__(kProbeThreads) probe_dfma(long long iters, double seed) {
    double acc[kChains];
    const double t = seed + threadIdx.x * 1e-9;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = t + c;
#pragma unroll 8
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("fma.rn.f64 %0, %1, %2, %0;" : "+d"(acc[c]) : "d"(0.9999999), "d"(1e-9));
    }
    double s = 0.0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    if (s == 1234567.0) g_probe_sink_d = s;
}

__global__ void __launch_bounds__(kProbeThreads) probe_dmma(long long iters, double seed) {
    constexpr int kMmaChains = 4;
    double d[kMmaChains][2];
    const double a = 0.9999999 + threadIdx.x * 1e-12, b = 1e-9 + seed;
#pragma unroll
    for (int c = 0; c < kMmaChains; ++c) { d[c][0] = seed + c; d[c][1] = seed - c; }
#pragma unroll 8
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kMmaChains; ++c)
            asm volatile("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0, %1}, {%2}, {%3}, {%0, %1};"
                         : "+d"(d[c][0]), "+d"(d[c][1])
                         : "d"(a), "d"(b));
    }
    double s = 0.0;
#pragma unroll
    for (int c = 0; c < kMmaChains; ++c) s += d[c][0] + d[c][1];
    if (s == 1234567.0) g_probe_sink_d = s;
}

}  // namespace
}  // namespace olc

extern "C" olc_status olc_debug_alu_rate(int kind, int64_t iters, void* stream, double* flops) {
    using namespace olc;
    if (!flops) return OLC_ERR_NULL;
    *flops = 0.0;
    if (kind < 0 || kind > 3 || iters < 1 || iters > (int64_t(1) << 40)) return OLC_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    const dim3 grid(sms * kProbeBlocksPerSm), block(kProbeThreads);
    const double threads = (double)grid.x * kProbeThreads;
    // flops one thread does per iteration
    const double per_iter = kind == 0 ? kChains * 4.0
                          : kind == 1 || kind == 2 ? kChains * 2.0
                          : 4 * (8.0 * 8.0 * 4.0 * 2.0) / 32.0;   // 4 MMAs per warp, per lane
    auto launch = [&](int64_t n) {
        switch (kind) {
            case 0: probe_ffma2<<<grid, block, 0, s>>>(n, 1.0f); break;
            case 1: probe_ffma<<<grid, block, 0, s>>>(n, 1.0f); break;
            case 2: probe_dfma<<<grid, block, 0, s>>>(n, 1.0); break;
            default: probe_dmma<<<grid, block, 0, s>>>(n, 1.0); break;
        }
        return cudaGetLastError();
    };
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    // warm-up at full length: module load, and the SM clock ramping up from
    // idle before the timed launch
    cudaError_t e = launch(iters);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = launch(iters);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return OLC_ERR_CUDA;
    }
    if (ms > 0.f) *flops = threads * per_iter * (double)iters / (ms * 1e-3);
    return OLC_OK;
}
