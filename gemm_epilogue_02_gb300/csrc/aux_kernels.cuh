// Small helper kernels around the fused GEMM.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace tgemm {

// Copy a [rows x cols] 16-bit matrix from pitch `lds` to pitch `ldd` (ldd a
// multiple of 8 elements, dst 16-byte aligned), so that tensor-memory-access
// copies, which need 16-byte row strides, can read an operand whose own pitch
// is unaligned.  Each thread writes one 16-byte vector of a destination row
// (8 elements) from 8 coalesced 2-byte source reads; blockIdx.y walks rows.
// HBM-bound: 2 x rows x cols x 2 bytes.
__global__ void __launch_bounds__(256) repack_rows_kernel(const uint16_t *__restrict__ src, long long lds,
                                                          uint16_t *__restrict__ dst, long long ldd,
                                                          long long rows, long long cols) {
    const long long vec_per_row = (cols + 7) / 8;
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const uint16_t *s = src + r * lds;
        uint4 *d = reinterpret_cast<uint4 *>(dst + r * ldd);
        for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < vec_per_row;
             v += static_cast<long long>(gridDim.x) * blockDim.x) {
            const long long c0 = v * 8;
            uint32_t w[4];
            if (c0 + 8 <= cols) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[i] = static_cast<uint32_t>(__ldg(s + c0 + 2 * i)) |
                           (static_cast<uint32_t>(__ldg(s + c0 + 2 * i + 1)) << 16);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t lo = (c0 + 2 * i < cols) ? __ldg(s + c0 + 2 * i) : 0u;
                    const uint32_t hi = (c0 + 2 * i + 1 < cols) ? __ldg(s + c0 + 2 * i + 1) : 0u;
                    w[i] = lo | (hi << 16);
                }
            }
            d[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// K == 0: the empty sum is 0, so C[i, j] = epi(bias[j]) (or epi(0)).
// act: 0 none, 1 ReLU, 2 GELU (the same activations as the fused kernel).
__global__ void fill_epilogue_kernel(const uint16_t *__restrict__ bias, uint16_t *__restrict__ C,
                                     long long ldc, int M, int N, int has_bias, int act,
                                     int is_bf16) {
    for (long long r = blockIdx.y; r < M; r += gridDim.y) {
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x) {
            float v = 0.0f;
            if (has_bias)
                v = is_bf16 ? __bfloat162float(__ushort_as_bfloat16(bias[j]))
                            : __half2float(__ushort_as_half(bias[j]));
            if (act == 1) v = (v <= 0.0f) ? 0.0f : v;
            if (act == 2) {
                const float u = 1.5957691216f * fmaf(0.044715f * v, v * v, v);
                v = v * __frcp_rn(1.0f + __expf(-u));
            }
            const uint16_t out = is_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                                         : __half_as_ushort(__float2half_rn(v));
            C[r * ldc + j] = out;
        }
    }
}

}  // namespace tgemm
