// Byte-level helper for moving 16-byte vectors between differently aligned
// places (the repacking of operands whose pitch is not a multiple of 16 bytes).
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

}  // namespace tgemm
