// Byte-level helpers for moving 16-byte vectors between differently aligned
// places (operand repacking, C rows whose pitch is not a multiple of 16 bytes).
#pragma once
#include <cstdint>

namespace tgemm {

// Bytes [o, o + 16) of the 32 bytes lo:hi (little-endian), o even, 0 < o < 16.
__device__ __forceinline__ uint4 shift_bytes16(const uint4 &lo, const uint4 &hi, int o) {
    uint32_t a0, a1, a2, a3, a4;
    switch (o >> 2) {       // whole words first
        case 0: a0 = lo.x; a1 = lo.y; a2 = lo.z; a3 = lo.w; a4 = hi.x; break;
        case 1: a0 = lo.y; a1 = lo.z; a2 = lo.w; a3 = hi.x; a4 = hi.y; break;
        case 2: a0 = lo.z; a1 = lo.w; a2 = hi.x; a3 = hi.y; a4 = hi.z; break;
        default: a0 = lo.w; a1 = hi.x; a2 = hi.y; a3 = hi.z; a4 = hi.w; break;
    }
    if (o & 2)              // then half a word
        return make_uint4(__funnelshift_r(a0, a1, 16), __funnelshift_r(a1, a2, 16), __funnelshift_r(a2, a3, 16),
                          __funnelshift_r(a3, a4, 16));
    return make_uint4(a0, a1, a2, a3);
}

// Bytes [start, start + 8) of the 16 bytes v (little-endian), 0 <= start < 16
// and even; bytes past the 16th read as zero, and the caller keeps the low
// bytes it needs.
__device__ __forceinline__ uint64_t bytes_at(const uint4 &v, int start) {
    const uint64_t lo = (static_cast<uint64_t>(v.y) << 32) | v.x;
    const uint64_t hi = (static_cast<uint64_t>(v.w) << 32) | v.z;
    if (start == 0) return lo;
    if (start >= 8) return hi >> (8 * (start - 8));
    return (lo >> (8 * start)) | (hi << (64 - 8 * start));
}

// Writes bytes [a, b) (a, b even, 0 <= a < b <= 16) of the 16-byte-aligned
// block at dst, taking the byte for position x from byte x + shift of v, in
// naturally aligned pieces of 8, 4 and 2 bytes (at most three stores).
__device__ __forceinline__ void store_bytes16(unsigned char *dst, const uint4 &v, int a, int b, int shift) {
    int x = a;
    while (x < b) {
        const int size = (x % 8 == 0 && x + 8 <= b) ? 8 : (x % 4 == 0 && x + 4 <= b) ? 4 : 2;
        const uint64_t bits = bytes_at(v, x + shift);
        if (size == 8) *reinterpret_cast<uint64_t *>(dst + x) = bits;
        else if (size == 4) *reinterpret_cast<uint32_t *>(dst + x) = static_cast<uint32_t>(bits);
        else *reinterpret_cast<uint16_t *>(dst + x) = static_cast<uint16_t>(bits);
        x += size;
    }
}

}  // namespace tgemm
