// Small helper kernels around the fused GEMM.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "bytes.cuh"
#include "debug_checks.cuh"
#include "ptx.cuh"

namespace tgemm {

// One 16-byte-aligned block of the source array at byte offset `off`: a
// single 16-byte load when the block lies inside the `span` bytes the matrix
// covers, else element by element (zero outside), so that no byte beyond the
// matrix is read.
__device__ __forceinline__ uint4 load_block16(const unsigned char *__restrict__ base, long long off,
                                              long long span) {
    if (off + 16 <= span) return __ldg(reinterpret_cast<const uint4 *>(base + off));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long e = off + 4 * i;
        const uint32_t lo = (e + 2 <= span) ? __ldg(reinterpret_cast<const uint16_t *>(base + e)) : 0u;
        const uint32_t hi = (e + 4 <= span) ? __ldg(reinterpret_cast<const uint16_t *>(base + e + 2)) : 0u;
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Copy a [rows x cols] 16-bit matrix from pitch `lds` to pitch `ldd` (ldd a
// multiple of 8 elements, dst 16-byte aligned; src 16-byte aligned), so that
// tensor-memory-access copies, which need 16-byte row strides, can read an
// operand whose own pitch is unaligned.  A source row starts o bytes past a
// 16-byte boundary (o even); each thread writes one 16-byte vector of a
// destination row (8 elements) from the two aligned 16-byte source blocks it
// straddles, shifted by o bytes.  The destination's pitch padding of the last
// vector is written as zero.  HBM-bound: 2 x rows x cols x 2 bytes.
// dst_elems (rows x ldd) and status serve the debug build's store check.
__global__ void __launch_bounds__(256) repack_rows_kernel(const uint16_t *__restrict__ src, long long lds,
                                                          uint16_t *__restrict__ dst, long long ldd,
                                                          long long rows, long long cols, long long dst_elems,
                                                          unsigned int *status) {
    // The fused kernel that reads dst may launch (and set itself up) now; it
    // waits for this grid's completion before its first global access.
    griddep_launch_dependents();
    const long long vec_per_row = (cols + 7) / 8;
    const unsigned char *base = reinterpret_cast<const unsigned char *>(src);
    const long long span = ((rows - 1) * lds + cols) * 2;   // bytes of src the matrix covers
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const long long row_off = r * lds * 2;
        const int o = static_cast<int>(row_off & 15);
        const long long al = row_off - o;
        uint4 *d = reinterpret_cast<uint4 *>(dst + r * ldd);
        for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < vec_per_row;
             v += static_cast<long long>(gridDim.x) * blockDim.x) {
            const uint4 lo = load_block16(base, al + 16 * v, span);
            uint4 out = lo;
            if (o != 0) out = shift_bytes16(lo, load_block16(base, al + 16 * v + 16, span), o);
            const long long valid = cols - 8 * v;   // elements of this vector inside the row (>= 1)
            if (valid < 8) {
                uint32_t w[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (2 * i >= valid) w[i] = 0u;
                    else if (2 * i + 1 >= valid) w[i] &= 0xFFFFu;
                }
                out = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (TGEMM_CHECK(r * ldd + 8 * v + 8 <= dst_elems, kChkRepack, status)) d[v] = out;
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
