// Device-side checks of the debug build (-DTGEMM_DEBUG, libtgemm_debug.so).
//
// The error classes the TileLang tutorial lists for hand-written kernels
// (out-of-bounds accesses, misaligned copies) are checked at every global
// access whose address the kernels compute: the innermost coordinate of each
// tensor-memory-access copy (it must start on a 16-byte boundary), and the
// element offset of each plain store of C, of each split-K partial and
// arrival counter, of the attention output and of the repacked operands,
// against bounds the host computes from the allocation sizes.  A failed check
// records TGEMM_ERR_DEBUG_CHECK in the device status word (unless another
// error is already there) and its check id in g_debug_check, and the access
// is skipped: nothing traps, and a skipped copy leaves its ring slot
// incomplete, which the bounded waits then end.  The release build compiles
// every check to `true`.
#pragma once
#include <cstdint>

namespace tgemm {

constexpr uint32_t kStatusDebugCheck = 8;   // TGEMM_ERR_DEBUG_CHECK

// Check ids (tgemm_debug_last_check).
enum DebugCheck : uint32_t {
    kChkTmaLoadA = 1,       // A's TMA load: innermost coordinate not 16-byte aligned
    kChkTmaLoadB = 2,       // B's TMA load: innermost coordinate not 16-byte aligned
    kChkTmaStoreC = 3,      // C's TMA store: coordinate negative, unaligned or past C's rows
    kChkStoreC = 4,         // masked store of C outside C's elements
    kChkPartial = 5,        // split-K partial outside the scratch
    kChkCounter = 6,        // arrival counter outside the counter buffer
    kChkAttnStore = 7,      // attention output store outside O's elements
    kChkRepack = 8,         // repack store outside the destination
};

// First check that failed since the host last read it (0: none).
__device__ unsigned int g_debug_check;

// Records a kernel error in the device status word.  Debug builds keep the
// first error since the host's last read (a copy skipped by a failed check
// later makes a wait run out, and that timeout must not hide the check);
// release builds keep the last one (a plain exchange: the compare-and-swap
// costs registers in the inlined waits).
__device__ __forceinline__ void record_status(unsigned int *status, uint32_t code) {
#ifdef TGEMM_DEBUG
    atomicCAS(status, 0u, code);
#else
    atomicExch(status, code);
#endif
}

#ifdef TGEMM_DEBUG
__device__ __noinline__ bool debug_fail(uint32_t id, unsigned int *status) {
    atomicCAS(status, 0u, kStatusDebugCheck);
    atomicCAS(&g_debug_check, 0u, id);
    return false;
}
#define TGEMM_CHECK(cond, id, status) ((cond) ? true : ::tgemm::debug_fail((id), (status)))
#else
#define TGEMM_CHECK(cond, id, status) true
#endif

}  // namespace tgemm
