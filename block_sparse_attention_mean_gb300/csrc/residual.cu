// residual.cu -- residual capture for sparse-attention residual compensation.
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "残差补偿找回被丢弃的尾部": the blocks a sparse mask drops carry small but nonzero
// attention mass, and the dense-minus-sparse residual changes across denoising
// steps less than the attention output does. So the residual is measured at an
// anchor step, R = O_dense - O_sparse, and later steps output O_sparse + R
// (bsa_forward_residual adds R in the forward's epilogue). This file holds the
// capture: an elementwise fp32 difference, HBM-bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace bsa {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// R[i] = float(dense[i]) - float(sparse[i]); four elements per thread and step
template <typename T>
__global__ void __launch_bounds__(256) residual_kernel(const T *__restrict__ dense, const T *__restrict__ sparse,
                                                       float *__restrict__ R, int64_t count)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < count; i += stride) {
        if (i + 4 <= count) {
            float4 r;
            r.x = to_f32(dense[i]) - to_f32(sparse[i]);
            r.y = to_f32(dense[i + 1]) - to_f32(sparse[i + 1]);
            r.z = to_f32(dense[i + 2]) - to_f32(sparse[i + 2]);
            r.w = to_f32(dense[i + 3]) - to_f32(sparse[i + 3]);
            *reinterpret_cast<float4 *>(R + i) = r;
        } else {
            for (int64_t k = i; k < count; ++k) R[k] = to_f32(dense[k]) - to_f32(sparse[k]);
        }
    }
}

}  // namespace

bsa_status launch_residual_capture(const void *dense, const void *sparse, int dt, int64_t count, float *R,
                                   cudaStream_t st)
{
    if (count == 0) return BSA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BSA_ERR_CUDA;
    const int64_t want = (count + 4 * 256 - 1) / (4 * 256);
    const int grid = static_cast<int>(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    if (dt == BSA_BF16)
        residual_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(dense),
                                                              static_cast<const __nv_bfloat16 *>(sparse), R, count);
    else
        residual_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(dense),
                                                       static_cast<const float *>(sparse), R, count);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace bsa
