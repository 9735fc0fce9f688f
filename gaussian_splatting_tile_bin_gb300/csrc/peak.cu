// peak.cu -- kernels of known arithmetic for measuring the device's FP32 and
// SFU lane-operation rates, the denominators of the raster kernels' roofline.
//
// Each thread keeps kChains independent dependency chains so that the pipe,
// not an instruction's latency, limits the rate, and the loop is unrolled so
// that the loop's own instructions take a small share of the issue slots.
// The result is stored only when it equals a value it cannot take in practice,
// which keeps the compiler from removing the work.
#include "internal.cuh"

namespace gsr {
namespace {

constexpr int kPeakChains = 16;
constexpr int kPeakUnroll = 8;
constexpr int kPeakThreads = 256;
constexpr int kPeakBlocksPerSM = 8;

// kChains fused multiply-adds per round: x = x a + b (a slightly below 1, so
// the values stay bounded).
__global__ void __launch_bounds__(kPeakThreads) k_peak_ffma(int rounds, float a, float b, float *__restrict__ sink)
{
    grid_dependency_begin();
    float x[kPeakChains];
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) x[k] = (float)threadIdx.x * 1e-3f + (float)k;
    for (int i = 0; i < rounds; i += kPeakUnroll) {
#pragma unroll
        for (int u = 0; u < kPeakUnroll; ++u)
#pragma unroll
            for (int k = 0; k < kPeakChains; ++k) x[k] = __fmaf_rn(x[k], a, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) s += x[k];
    if (s == -1234.5f) sink[0] = s;
}

// kChains base-2 exponentials per round on the SFU (the instruction the raster
// kernels' exponential is built on): x = 2^-x keeps every value in (0, 1].
__global__ void __launch_bounds__(kPeakThreads) k_peak_ex2(int rounds, float *__restrict__ sink)
{
    grid_dependency_begin();
    float x[kPeakChains];
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) x[k] = (float)threadIdx.x * 1e-3f + (float)k * 0.01f;
    for (int i = 0; i < rounds; i += kPeakUnroll) {
#pragma unroll
        for (int u = 0; u < kPeakUnroll; ++u)
#pragma unroll
            for (int k = 0; k < kPeakChains; ++k) {
                float y;
                asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-x[k]));
                x[k] = y;
            }
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) s += x[k];
    if (s == -1234.5f) sink[0] = s;
}

}  // namespace

int peak_kernel(gsr_ctx *ctx, int kind, int32_t iters, float *sink, uint64_t *lane_ops, cudaStream_t stream)
{
    const int rounds = (iters + kPeakUnroll - 1) / kPeakUnroll * kPeakUnroll;
    const int blocks = ctx->num_sms * kPeakBlocksPerSM;
    *lane_ops = (uint64_t)blocks * kPeakThreads * (uint64_t)rounds * kPeakChains;
    const cudaError_t e =
        kind == GSR_PEAK_FFMA
            ? launch_kernel(ctx, k_peak_ffma, dim3(blocks), dim3(kPeakThreads), stream, rounds, 0.99993f, 1e-4f, sink)
            : launch_kernel(ctx, k_peak_ex2, dim3(blocks), dim3(kPeakThreads), stream, rounds, sink);
    return cuda_check(ctx, e, "peak kernel launch");
}

}  // namespace gsr
