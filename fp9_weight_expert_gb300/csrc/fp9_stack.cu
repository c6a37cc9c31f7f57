// Stack glue between MoE layers: h += y, then x = RMSNorm(h) with unit gain.
//
// The pages keep the norm and the residual add on the GPU side of each
// decode layer, next to attention ("第 9 章 MTP1 dual-lane overlap", section
// 9.5: stage0 holds layernorm and the residual add); the step between two
// MoE layers of a stack is h <- h + MoE(RMSNorm(h)).
#include <cuda_runtime.h>

#include <cstdint>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9moe.h"

namespace fp9 {

// One CTA per token; each thread keeps its float4 columns in a fixed order,
// and the block sum of squares is added in a fixed order.
__global__ void __launch_bounds__(kNormThreads) residual_rmsnorm_kernel(float* h, const float* y, float* x_out,
                                                                       int64_t H, float eps) {
    __shared__ float red[kNormThreads / 32];
    __shared__ float s_scale;
    grid_dependency_wait();  // y and h are complete
    grid_launch_dependents();
    const int t = blockIdx.x;
    float4* h4 = reinterpret_cast<float4*>(h + t * H);
    const float4* y4 = y ? reinterpret_cast<const float4*>(y + t * H) : nullptr;
    float4* x4 = reinterpret_cast<float4*>(x_out + t * H);
    const int64_t H4 = H / 4;
    float ss = 0.0f;
    for (int64_t c = threadIdx.x; c < H4; c += kNormThreads) {
        const float4 v = residual4(h4, y4, c);
        if (y4) h4[c] = v;
        ss = sumsq4(v, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) s_scale = rms_scale(red, H, eps);
    __syncthreads();
    const float scale = s_scale;
    for (int64_t c = threadIdx.x; c < H4; c += kNormThreads) {
        const float4 v = h4[c];
        x4[c] = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    }
}

}  // namespace fp9

using namespace fp9;

extern "C" fp9_status fp9_residual_rmsnorm(float* h, const float* y, float* x_out, int32_t bsz, int64_t hidden,
                                           float eps, void* stream) {
    FP9_CHECK_ARG(h != nullptr && x_out != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(bsz >= 1 && bsz <= FP9_MAX_BSZ, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(hidden >= 4 && hidden % 4 == 0, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(eps >= 0.0f, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(h, 16) && aligned(x_out, 16) && (y == nullptr || aligned(y, 16)), FP9_ERR_ALIGN);
    FP9_CUDA_TRY(launch_pdl(residual_rmsnorm_kernel, dim3(bsz), dim3(kNormThreads), 0,
                            static_cast<cudaStream_t>(stream), h, y, x_out, hidden, eps));
    return FP9_OK;
}
