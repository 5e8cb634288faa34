// sv_check.cuh -- range checks of the kernels' memory accesses, compiled in with -DSV_DEBUG.
//
// A debug build checks the index of every global-memory access the kernels make against the
// extent of the array it falls in.  An index out of range is recorded (the first one: its site
// number and the index, in this translation unit's debug word, which spec_verify_debug_fault
// reads back) and the access is skipped; nothing traps and nothing asserts, so the context stays
// usable and the host reads what happened.  In a release build every check is the constant true
// and compiles away.
#pragma once

#include <stdint.h>

namespace sv {

#ifdef SV_DEBUG
// First range violation of this module: bit 63 set, site number in bits 48..62, the low 48 bits
// of the offending index.  Zero while nothing has gone out of range.
static __device__ unsigned long long g_sv_debug_fault;

__device__ __forceinline__ bool debug_in_range(int64_t i, int64_t n, int site)
{
    if (i >= 0 && i < n) return true;
    const unsigned long long w = (1ull << 63) | ((unsigned long long)(site & 0x7fff) << 48) |
                                 ((unsigned long long)i & 0xffffffffffffull);
    atomicCAS(&g_sv_debug_fault, 0ull, w);
    return false;
}
#define SV_INB(i, n, site) ::sv::debug_in_range((int64_t)(i), (int64_t)(n), (site))
#else
#define SV_INB(i, n, site) true
#endif

}  // namespace sv
