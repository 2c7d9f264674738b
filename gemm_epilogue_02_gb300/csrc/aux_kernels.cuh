// Small helper kernels around the fused GEMM.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace tgemm {

// Copy a [rows x cols] 16-bit matrix from pitch `lds` to pitch `ldd` (ldd a
// multiple of 8 elements), so that tensor-memory-access copies, which need
// 16-byte row strides, can read an operand whose own pitch is unaligned.
__global__ void repack_rows_kernel(const uint16_t *__restrict__ src, long long lds,
                                   uint16_t *__restrict__ dst, long long ldd, long long rows,
                                   long long cols) {
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const uint16_t *s = src + r * lds;
        uint16_t *d = dst + r * ldd;
        for (long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; c < cols;
             c += static_cast<long long>(gridDim.x) * blockDim.x)
            d[c] = s[c];
    }
}

// K == 0: the empty sum is 0, so C[i, j] = epi(bias[j]) (or epi(0)).
__global__ void fill_epilogue_kernel(const uint16_t *__restrict__ bias, uint16_t *__restrict__ C,
                                     long long ldc, int M, int N, int has_bias, int relu,
                                     int is_bf16) {
    for (long long r = blockIdx.y; r < M; r += gridDim.y) {
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x) {
            float v = 0.0f;
            if (has_bias)
                v = is_bf16 ? __bfloat162float(__ushort_as_bfloat16(bias[j]))
                            : __half2float(__ushort_as_half(bias[j]));
            if (relu) v = (v <= 0.0f) ? 0.0f : v;
            const uint16_t out = is_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                                         : __half_as_ushort(__float2half_rn(v));
            C[r * ldc + j] = out;
        }
    }
}

}  // namespace tgemm
