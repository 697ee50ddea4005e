// sb_debug.cu -- test hooks that expose device helpers of the projection kernels.
#include <cstdint>

#include "sb.h"
#include "sb_combine_math.cuh"
#include "sb_gumbel.cuh"

namespace {

__global__ void gumbel_from_bits_kernel(const uint32_t *b, float *g, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) g[i] = sb::gumbel_from_bits(b[i] & 0xFFFFFFu);
}

__global__ void combine_math_kernel(int op, const float *x, float *y, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) y[i] = op == 0 ? sb::exp_nonpos(x[i]) : sb::log_sum(x[i]);
}

}  // namespace

extern "C" int32_t sb_debug_combine_math(int32_t op, const float *x, float *y, int64_t count,
                                         void *stream) {
    if ((op != 0 && op != 1) || !x || !y || count < 1 || count > (int64_t(1) << 31))
        return SB_ERR_INVALID_ARG;
    const int threads = 256;
    const int64_t blocks = (count + threads - 1) / threads;
    combine_math_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                          static_cast<cudaStream_t>(stream)>>>(op, x, y, count);
    return cudaGetLastError() == cudaSuccess ? SB_OK : SB_ERR_CUDA;
}

extern "C" int32_t sb_debug_gumbel_from_bits(const uint32_t *bits, float *g, int64_t count,
                                             void *stream) {
    if (!bits || !g || count < 1 || count > (int64_t(1) << 31)) return SB_ERR_INVALID_ARG;
    const int threads = 256;
    const int64_t blocks = (count + threads - 1) / threads;
    gumbel_from_bits_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                              static_cast<cudaStream_t>(stream)>>>(bits, g, count);
    return cudaGetLastError() == cudaSuccess ? SB_OK : SB_ERR_CUDA;
}
